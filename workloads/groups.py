"""Parameter groups of the benchmark workloads (shapes only).

Sources for the shapes: the TIDE abstract names Llama-3.1 70B, Wan2.2 and Qwen3-30B-A3B as its
training workloads; Tables 7 and 8 of the figure/table list measure 32 MiB and 128 MiB per-rank
shards.  The layer shapes below are those models' public decoder-layer / DiT-block shapes.
"""
from __future__ import annotations

import dataclasses
from typing import List, Tuple

Param = Tuple[str, int, int]  # (name, rows = dim 0, row_len = product of the other dims)


@dataclasses.dataclass(frozen=True)
class Group:
    """One FSDP parameter group sharded over ``R`` emulated ranks.

    ``grad_kind`` says how the bf16 gradients are drawn: ``"int"`` = integers uniform in
    ``[-8, 8]`` (all 17 values), ``"normal"`` = N(0, ``grad_sigma``) stand-in.  The all-gather
    input shards are always the N(0, ``shard_sigma``) stand-in.  ``grad_seed_per_rank`` picks
    seed ``r`` for rank ``r``; otherwise every rank uses ``grad_seed`` (with the rank as the
    stream index).
    """

    name: str
    R: int
    params: Tuple[Param, ...]
    grad_kind: str = "normal"
    grad_sigma: float = 1e-3
    shard_sigma: float = 0.02
    grad_seed: int = 0
    grad_seed_per_rank: bool = True
    shard_seed_base: int = 1000

    @property
    def P(self) -> int:
        return len(self.params)

    @property
    def rows(self) -> List[int]:
        return [p[1] for p in self.params]

    @property
    def row_len(self) -> List[int]:
        return [p[2] for p in self.params]

    def numel(self, p: int) -> int:
        """Element count of parameter ``p`` (unsharded)."""
        return self.params[p][1] * self.params[p][2]

    def grad_seed_of(self, r: int) -> int:
        return r if self.grad_seed_per_rank else self.grad_seed

    def shard_seed_of(self, r: int) -> int:
        return self.shard_seed_base + r

    def with_R(self, R: int, name: str | None = None) -> "Group":
        return dataclasses.replace(self, R=R, name=name or f"{self.name}_R{R}")

    def scaled(self, div: int, name: str | None = None) -> "Group":
        """Same parameter list with every dimension divided by ``div`` (at least 1).

        Keeps the parameter count and order, so reduced-size parity cases still cover
        every segment kind of the full group (padding, empty ranks, tiny norms)."""
        ps = tuple((n, max(1, r // div), max(1, l // div)) for (n, r, l) in self.params)
        return dataclasses.replace(self, params=ps, name=name or f"{self.name}_div{div}")


def tiny_group() -> Group:
    """R=4, three parameters (5,3), (7,4), (2,6); integer gradients in [-8, 8], seed 0."""
    return Group(
        name="tiny",
        R=4,
        params=(("a", 5, 3), ("b", 7, 4), ("c", 2, 6)),
        grad_kind="int",
        grad_seed=0,
        grad_seed_per_rank=False,
    )


def llama8b_layer() -> Group:
    """Llama-3.1-8B decoder layer, R=8."""
    h, kv, f = 4096, 1024, 14336
    ps = (
        ("q", h, h), ("k", kv, h), ("v", kv, h), ("o", h, h),
        ("gate", f, h), ("up", f, h), ("down", h, f),
        ("input_norm", h, 1), ("post_norm", h, 1),
    )
    return Group(name="llama3.1-8b-layer", R=8, params=ps)


def qwen3_moe_layer() -> Group:
    """Qwen3-30B-A3B MoE layer, R=8: attention, router, 128 experts (gate, up, down), two norms."""
    ps: List[Param] = [
        ("q", 4096, 2048), ("k", 512, 2048), ("v", 512, 2048), ("o", 2048, 4096),
        ("q_norm", 128, 1), ("k_norm", 128, 1), ("router", 128, 2048),
    ]
    for e in range(128):
        ps += [(f"e{e}.gate", 768, 2048), (f"e{e}.up", 768, 2048), (f"e{e}.down", 2048, 768)]
    ps += [("input_norm", 2048, 1), ("post_norm", 2048, 1)]
    return Group(name="qwen3-30b-a3b-moe-layer", R=8, params=tuple(ps))


def llama70b_layer() -> Group:
    """Llama-3.1-70B decoder layer, R=8."""
    h, kv, f = 8192, 1024, 28672
    ps = (
        ("q", h, h), ("k", kv, h), ("v", kv, h), ("o", h, h),
        ("gate", f, h), ("up", f, h), ("down", h, f),
        ("input_norm", h, 1), ("post_norm", h, 1),
    )
    return Group(name="llama3.1-70b-layer", R=8, params=ps)


# Wan2.2-14B DiT block (dim 5120, ffn 13824) cycled after one extra 5119x5120 matrix until the
# next whole parameter would overflow a 32 MiB (8,388,608 fp32 elements) per-rank shard, then
# topped up by one 1-D filler parameter of R x (remaining elements).  The lists are written out
# here; a test recomputes each per-rank shard size with the oracle's planner.
_WAN_CYCLE: Tuple[Param, ...] = (
    ("self.q", 5120, 5120), ("self.k", 5120, 5120), ("self.v", 5120, 5120), ("self.o", 5120, 5120),
    ("cross.q", 5120, 5120), ("cross.k", 5120, 5120), ("cross.v", 5120, 5120), ("cross.o", 5120, 5120),
    ("ffn.0", 13824, 5120), ("ffn.2", 5120, 13824), ("modulation", 6, 5120),
    ("norm.a", 5120, 1), ("norm.b", 5120, 1),
)
_WAN_EXTRA: Param = ("extra", 5119, 5120)
# number of cycle entries taken before the filler, and the filler's total element count
_WAN_FILL = {8: (1, 14_680_064), 16: (4, 3_145_728), 32: (8, 32_505_856), 64: (19, 1_759_232)}
WAN_SHARD_ELEMS = 8_388_608


def wan_sweep_group(R: int) -> Group:
    """Wan2.2-14B-shaped block repeated to a 32 MiB fp32 shard per rank, R in {8, 16, 32, 64}."""
    ncyc, filler = _WAN_FILL[R]
    ps = [_WAN_EXTRA]
    for i in range(ncyc):
        n, r, l = _WAN_CYCLE[i % len(_WAN_CYCLE)]
        ps.append((f"{n}#{i // len(_WAN_CYCLE)}", r, l))
    ps.append(("filler", filler, 1))
    return Group(name=f"wan2.2-sweep-R{R}", R=R, params=tuple(ps))


GROUPS = {
    "tiny": tiny_group,
    "llama8b": llama8b_layer,
    "qwen3moe": qwen3_moe_layer,
    "llama70b": llama70b_layer,
    "wan_r8": lambda: wan_sweep_group(8),
    "wan_r16": lambda: wan_sweep_group(16),
    "wan_r32": lambda: wan_sweep_group(32),
    "wan_r64": lambda: wan_sweep_group(64),
}


def group(name: str) -> Group:
    return GROUPS[name]()
