"""OSCAR INT2 paged-KV decode hot path for one GB300 GPU (sm_103a).

liboscar (C ABI, include/oscar.h) holds the pool and the CUDA kernels; ``binding`` is a ctypes
binding with the same names; ``Pool`` wraps it with PyTorch tensors for device memory and streams.
"""
from .binding import OscarConfig, OscarError, lib, oscar_version  # noqa: F401
from .pool import Pool  # noqa: F401
