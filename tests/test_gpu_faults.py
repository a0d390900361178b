"""Fault injection on the host into the pool's INT2 path: a page-table entry set out of range
through oscar_debug_set_page_entry. The kernels that read it must report OSCAR_DEVERR_PAGE through
the device error word, touch nothing outside the pool (the decode substitutes an in-bounds page,
the demote skips its write), and the pool must decode correctly again once the entry is restored.
Nothing here faults a GPU: every injected id is caught by a range check before any access."""
import numpy as np
import pytest
import torch

from bit_kv_cache_paged_gb300 import binding as B
from harness import Case, bits_to_dev


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _expect_page_error(pool):
    with pytest.raises(B.OscarError) as e:
        pool.check()
    assert e.value.status == B.OSCAR_EDEVICE and e.value.detail & B.DEVERR_PAGE
    pool.check()  # the word was cleared


@pytest.mark.gpu
def test_corrupt_int2_page_entry_in_decode_then_clean_step_matches_oracle():
    max_pages = 2 * 70
    c = Case(layers=2, Hq=8, Hkv=2, max_seqs=2, max_len=4200, max_pages=max_pages)
    c.add(0)
    c.add(1)
    c.step([0, 1], [1500, 2600])
    ids = [0, 1]
    for bad in (-1, max_pages, 2 ** 31 - 1):
        B.oscar_debug_set_page_entry(c.pool.handle, 1, 3, bad, _stream())
        c.pool.step_begin(ids, [0, 0])
        q = bits_to_dev(c.q_bits(0, ids), (2, c.Hq, 128))
        out = c.pool.attend(1, q)
        torch.cuda.synchronize()
        _expect_page_error(c.pool)
        assert out.shape == (2, c.Hq, 128)
        B.oscar_debug_restore_page_table(c.pool.handle, 1, _stream())
    # a clean step afterwards: both sequences, both layers, match the fp64 oracle
    c.step(ids, [1, 1])
    for layer in (0, 1):
        c.check_decode(layer, 1, ids)


@pytest.mark.gpu
def test_corrupt_int2_page_entry_in_demote_is_reported():
    """The tail page's entry is out of range when the step's demote writes into it: the demote
    reports the page error and writes nothing; the other sequence of the batch is unaffected."""
    c = Case(layers=1, Hq=4, Hkv=1, max_seqs=2, max_len=4000, max_pages=2 * 64)
    c.add(0)
    c.add(1)
    c.step([0, 1], [2600, 2000])
    L, F, n_pages = c.pool.seq_info(0)
    assert (F - 64) % 64 != 0  # the next demoted token lands in the existing tail page
    B.oscar_debug_set_page_entry(c.pool.handle, 0, n_pages - 1, 1 << 30, _stream())
    before = c.pool.debug_read_int2(1, 0, 0, 64, c.pool.seq_info(1)[1] - 64)
    c.step([0, 1], [1, 1])
    torch.cuda.synchronize()
    _expect_page_error(c.pool)
    B.oscar_debug_restore_page_table(c.pool.handle, 0, _stream())
    after = c.pool.debug_read_int2(1, 0, 0, 64, len(before[0]))
    for x, y in zip(before, after):
        assert torch.equal(x, y)
    # sequence 1 still decodes correctly in the same pool (sequence 0 holds one unwritten row)
    c.step([1], [1])
    c.check_decode(0, 2, [1])


@pytest.mark.gpu
def test_misaligned_buffers_are_refused_before_any_launch():
    """The step calls read and write their device buffers in 16-byte pieces: a base that is not
    16-byte aligned is refused with OSCAR_EINVAL and nothing is launched."""
    c = Case(layers=1, Hq=4, Hkv=1, max_seqs=1, max_len=2000)
    c.add(0)
    c.pool.step_begin([0], [300])
    n = 300 * c.Hkv * 128
    buf = torch.zeros(2 * n + 8, dtype=torch.bfloat16, device="cuda")
    k_bad, v_bad = buf[1:1 + n], buf[n + 2:2 * n + 2]  # 2-byte offsets
    assert k_bad.data_ptr() % 16 != 0 and v_bad.data_ptr() % 16 != 0
    launches = B.oscar_launch_count(c.pool.handle)
    with pytest.raises(B.OscarError) as e:
        B.oscar_append_and_demote(c.pool.handle, 0, k_bad, v_bad, _stream())
    assert e.value.status == B.OSCAR_EINVAL
    # the other step calls check their buffers the same way
    q = torch.zeros(c.Hq * 128 + 8, dtype=torch.bfloat16, device="cuda")
    q_rot = torch.zeros(c.Hq * 128 + 4, dtype=torch.float32, device="cuda")
    parts = torch.zeros(B.oscar_partials_bytes(c.pool.handle, 1) + 16, dtype=torch.uint8, device="cuda")
    calls = (lambda: B.oscar_rotate_q(c.pool.handle, 0, q[1:], q_rot, _stream()),
             lambda: B.oscar_decode(c.pool.handle, 0, q, q_rot[1:], parts, _stream()),
             lambda: B.oscar_merge(c.pool.handle, 0, parts[8:], q_rot, _stream()),
             lambda: B.oscar_merge(c.pool.handle, 0, parts, q_rot[2:], _stream()))
    for call in calls:
        with pytest.raises(B.OscarError) as e:
            call()
        assert e.value.status == B.OSCAR_EINVAL
    assert B.oscar_launch_count(c.pool.handle) == launches
    c.pool.check()
