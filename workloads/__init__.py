"""Synthetic parameter groups and seeded input bits for the TIDE reduce-scatter / all-gather path.

This package is shared by the CPU oracle's tests and the GPU harness.  It only *names* shapes and
*draws* bits; it holds none of the sharding, padding, offset or reduction arithmetic, which the
oracle and the CUDA library each implement on their own.

A group is ``R`` emulated ranks plus an ordered list of parameters.  Each parameter is given as
``(name, rows, row_len)``: ``rows`` is dim 0 (the sharded dim) and ``row_len`` is the product of the
remaining dims (1 for a 1-D tensor).  The layer shapes follow the models named in the TIDE abstract
(Llama-3.1 70B, Wan2.2, Qwen3-30B-A3B) and the 32 MiB reduce-scatter output of its Tables 7 and 8.
"""
from .groups import Group, GROUPS, group, tiny_group, wan_sweep_group  # noqa: F401
from .rng import (  # noqa: F401
    grad_bits,
    group_grads,
    normal_bf16_bits,
    shard_bits,
    stream_key,
    uniform_int_bf16_bits,
)
