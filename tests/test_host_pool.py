"""CPU tests of liboscar's C ABI: the library loads and exports every symbol the header declares,
and the host-side pool logic (zones, page allocation, prefix sharing, capacity errors, storage
accounting) behaves as specified. No compute calls: pools are created with OSCAR_FLAG_HOST_ONLY."""
import ctypes

import pytest

import oracle as O
from bit_kv_cache_paged_gb300 import binding as B
from bit_kv_cache_paged_gb300 import build as BLD
from bit_kv_cache_paged_gb300.pool import Pool


@pytest.fixture(scope="module", autouse=True)
def built():
    BLD.build()
    return B.lib()


def test_exports_every_header_symbol():
    names = B.header_symbols()
    assert len(names) >= 20
    L = ctypes.CDLL(BLD.LIB)
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    assert set(names) == set(B._SIGS), "binding and header disagree"
    assert "sm_103a" in B.oscar_version()


def cfg(**kw):
    c = dict(num_layers=2, num_q_heads=32, num_kv_heads=8, max_seqs=8, max_seq_len=40000,
             max_int2_pages=2000)
    c.update(kw)
    return c


def host_pool(**kw):
    return Pool(**cfg(**kw), host_only=True)


def test_invalid_configs_rejected():
    for bad in (dict(num_q_heads=24), dict(num_q_heads=8, num_kv_heads=8), dict(group_size=64),
                dict(max_int2_pages=0), dict(max_seqs=0)):
        c = cfg(**bad)
        oc = B.OscarConfig(c["num_layers"], c["num_q_heads"], c["num_kv_heads"], 128, 64, 64, 256,
                           bad.get("group_size", 128), c["max_seqs"], c["max_seq_len"], c["max_int2_pages"], 0, 0)
        assert B.oscar_arena_bytes(oc) == 0
    oc = B.OscarConfig(1, 4, 1, 64, 64, 64, 256, 128, 1, 100, 1, 0, 0)  # head_dim 64
    assert B.oscar_arena_bytes(oc) == 0


def test_arena_bytes_cover_int2_pool():
    oc = B.OscarConfig(36, 32, 8, 128, 64, 64, 256, 128, 32, 100100, 51200, 0, 0)
    n = B.oscar_arena_bytes(oc)
    int2 = 36 * 51200 * 8 * 4608
    bf16 = 36 * (32 * 8 * 64 * 128 * 2 * 2 + 32 * 8 * 256 * 128 * 2 * 2)
    assert int2 + bf16 < n < int2 + bf16 + 200 * 2 ** 20
    oc32 = B.OscarConfig(1, 4, 1, 128, 64, 64, 256, 32, 1, 4096, 10, 0, 0)
    oc128 = B.OscarConfig(1, 4, 1, 128, 64, 64, 256, 128, 1, 4096, 10, 0, 0)
    assert B.oscar_arena_bytes(oc32) - B.oscar_arena_bytes(oc128) >= 10 * (6144 - 4608)


@pytest.mark.parametrize("L", [1, 63, 64, 65, 300, 320, 321, 384, 385, 2048, 32768])
def test_zones_and_pages_match_oracle(L):
    p = host_pool()
    p.seq_add(0)
    p.step_begin([0], [L])
    Lg, F, npg = p.seq_info(0)
    _, F_ref = O.zone_bounds(L)
    assert (Lg, F) == (L, F_ref)
    assert npg == (max(0, F_ref - 64) + 63) // 64


def test_decode_steps_advance_frontier_and_pages():
    p = host_pool()
    p.seq_add(3)
    p.step_begin([3], [320])
    assert p.seq_info(3) == (320, 64, 0)
    for k in range(1, 130):
        p.step_begin([3], [1])
        L, F, npg = p.seq_info(3)
        assert L == 320 + k and F == 64 + k and npg == (k + 63) // 64
    assert p.stats()["int2_pages_used"] == 3


def test_prefix_sharing_refcounts_pages():
    p = host_pool()
    p.seq_add(0)
    p.step_begin([0], [32768 + 256])
    used = p.stats()["int2_pages_used"]
    assert used == 511  # [64, 32768) is 511 full pages
    p.seq_add(1, 0, 32768)
    assert p.seq_info(1) == (32768, 32768, 511)
    assert p.stats()["int2_pages_used"] == used  # shared, not copied
    assert p.stats()["sink_pages_used"] == 1
    p.step_begin([1], [1000])
    L, F, npg = p.seq_info(1)
    assert (L, F) == (33768, 33768 - 256) and npg == 511 + (F - 32768 + 63) // 64
    p.seq_remove(0)  # the prefix pages stay alive through seq 1
    assert p.stats()["int2_pages_used"] == npg
    p.seq_remove(1)
    assert p.stats()["int2_pages_used"] == 0 and p.stats()["sink_pages_used"] == 0


def test_share_requires_demoted_aligned_prefix():
    p = host_pool()
    p.seq_add(0)
    p.step_begin([0], [5000])
    with pytest.raises(B.OscarError):
        p.seq_add(1, 0, 5000)          # not yet demoted (frontier 4744)
    with pytest.raises(B.OscarError):
        p.seq_add(1, 0, 64 + 64 * 10 + 5)  # not page aligned
    p.seq_add(1, 0, 64 + 64 * 10)


def test_capacity_error_rolls_back():
    p = host_pool(max_int2_pages=10)
    p.seq_add(0)
    p.step_begin([0], [64 + 256 + 640])  # exactly 10 pages
    with pytest.raises(B.OscarError) as e:
        p.step_begin([0], [1])
    assert e.value.status == B.OSCAR_EFULL
    assert p.seq_info(0) == (960, 704, 10)
    p.seq_add(1)
    p.step_begin([1], [320])  # no INT2 pages needed
    p.seq_remove(0)
    p.step_begin([1], [64])
    assert p.seq_info(1)[2] == 1


def test_bad_arguments():
    p = host_pool()
    p.seq_add(0)
    for args in (([5], [1]), ([0, 0], [1, 1]), ([0], [-1]), ([0], [10 ** 6])):
        with pytest.raises(B.OscarError):
            p.step_begin(*args)
    with pytest.raises(B.OscarError):
        p.seq_add(0)
    with pytest.raises(B.OscarError):
        p.seq_remove(7)
    # launches on a host-only pool are refused
    with pytest.raises(B.OscarError):
        B.oscar_rotate_q(p.handle, 0, 1, 1, None)


def test_storage_bits_per_element_match_pages():
    """Pool bytes per token reproduce the pages' bits-per-element figures (2.28 at 128K, 2.38 at 32K)."""
    p = host_pool(num_layers=1, num_kv_heads=1, num_q_heads=4)
    st = p.stats()
    per_elem_bf16 = st["bf16_bytes_per_token"] * 8 / (2 * 128)
    per_elem_int2 = st["int2_bytes_per_token"] * 8 / (2 * 128)
    assert per_elem_bf16 == 16 and per_elem_int2 == 2.25
    for L, want in ((131072, 2.28), (32768, 2.38)):
        bpe = (320 * per_elem_bf16 + (L - 320) * per_elem_int2) / L
        assert round(bpe, 2) == want
        assert abs(bpe - O.bits_per_element(L)) < 1e-12


def test_config_flags_are_validated():
    """Unknown flag bits make the config invalid; the Lloyd-Max flag is accepted."""
    from bit_kv_cache_paged_gb300 import binding as B
    base = dict(num_layers=1, num_q_heads=4, num_kv_heads=1, head_dim=128, page_size=64, sink_size=64,
                recent_size=256, group_size=128, max_seqs=2, max_seq_len=1000, max_int2_pages=32, v_rot_absorbed=0)
    assert B.oscar_arena_bytes(B.OscarConfig(**base, flags=B.OSCAR_FLAG_LLOYD_MAX)) > 0
    assert B.oscar_arena_bytes(B.OscarConfig(**base, flags=0x4)) == 0


def _int2_workers(p):
    """INT2 decode workers of the current step."""
    return p.int2_workers()


def test_partials_bound_depends_on_batch_only():
    """The partials size is a bound of the batch (BF16 slot per pair, at most 64 INT2 workers per
    pair plus one segment per pair), the same for every step of that batch."""
    p = host_pool(max_seqs=8, max_seq_len=40000, max_int2_pages=8000)
    p.seq_add(0)
    slot = p.Hq // p.Hkv * (2 + 128) * 4
    sizes = set()
    for n in (400, 1, 64, 32000):
        p.step_begin([0], [n])
        sizes.add(p.partials_bytes())
        assert p.partials_bytes() >= (p.int2_workers() + 2 * p.Hkv) * slot
    assert sizes == {(8 * 64 + 2 * 8) * slot}


def test_decode_worker_count_rule():
    """Workers = clamp(ceil(units / 4), 1, resident maximum), and at most 64 per (sequence, KV
    head) on average so that a step with few rows leaves the merge few partials."""
    p = host_pool(max_seqs=8, max_seq_len=40000, max_int2_pages=8000)
    p.seq_add(0)
    p.step_begin([0], [32768])  # 8 KV heads x 507 pages = 4056 units: the cap (8 x 64) binds
    assert p.seq_info(0)[2] == 507
    assert _int2_workers(p) == 8 * 64
    q = host_pool()
    q.seq_add(0)
    q.step_begin([0], [2048])  # 8 x 27 = 216 units: 4 pages per worker binds
    assert q.seq_info(0)[2] == 27
    assert _int2_workers(q) == 216 // 4
    r = host_pool(max_seqs=8, max_seq_len=40000, max_int2_pages=8000)
    for s in range(8):
        r.seq_add(s)
    r.step_begin(list(range(8)), [32768] * 8)  # 32448 units, cap 4096: the resident maximum binds
    assert _int2_workers(r) == 152 * 12  # a host-only pool assumes 152 SMs x 12 workers
