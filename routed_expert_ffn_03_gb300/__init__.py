"""Decode-time routed Mixture-of-Experts layer for GB300 (sm_103a).

The compute path is the C ABI of include/moe.h, implemented by hand-written CUDA kernels
in ``csrc/`` and built in-tree into ``libmoe.so``; ``moe`` is its Python binding.
"""
from .moe import (Config, Context, FileTier, MoeError, Stats, expert_blob_bytes, lib, route_noalloc,  # noqa: F401
                  rvq_block_split,
                  strerror, ROUTER_SOFTMAX, ROUTER_SIGMOID, W_RVQ3, W_INT4,
                  OK, EINVAL, ENOMEM, EBUDGET, ECUDA, ESTATE, ETIMEOUT, ENOTFOUND, EIO)
