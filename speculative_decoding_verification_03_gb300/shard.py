"""A verification batch sharded over GPUs, one process per GPU.

The B sequences of a step are independent ("Speculative Decoding: Draft,
EAGLE, MTP", section "one speculative step": each sequence's acceptance walk
reads only its own rows), so each rank verifies a contiguous block of them
with no exchange.  The AV refit is the one step that spans the batch: its
round update solves one system from gradient and Hessian sums over every
label of the round ("Adaptive Verification without a confidence head",
section "Fitting the coefficients").  The sums are additive, so each rank
accumulates its own sequences (round_len = 0), the ranks sum the 4K + 2
fp64 accumulator values with one all-reduce, and every rank then solves the
same system and applies the same update to its copy of theta.

Host logic only: the accumulation and the solve run in the library's
kernels (binding.AVState), the sum in torch.distributed.
"""
from __future__ import annotations

import numpy as np


def shard_range(B: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous block [b0, b1) of the B sequences that `rank` of `world`
    verifies: sizes differ by at most one, lower ranks take the extra ones."""
    if world < 1 or not 0 <= rank < world or B < 0:
        raise ValueError("bad shard request")
    base, extra = divmod(B, world)
    b0 = rank * base + min(rank, extra)
    return b0, b0 + base + (1 if rank < extra else 0)


def block_layout(K: int) -> dict:
    """Slices of the accumulator block (sv_av_accum_bytes): g (slope first,
    then the K intercepts), H_ww, H_wb[K], H_bb[K], n[K]."""
    return dict(g=slice(0, K + 1), Hww=slice(K + 1, K + 2), Hwb=slice(K + 2, 2 * K + 2),
                Hbb=slice(2 * K + 2, 3 * K + 2), n=slice(3 * K + 2, 4 * K + 2))


def block_from_dense(g, H, n) -> np.ndarray:
    """The block of an arrow-shaped system given densely (g [K+1],
    H [K+1][K+1] with index 0 the slope, n [K])."""
    g, H, n = np.asarray(g, np.float64), np.asarray(H, np.float64), np.asarray(n, np.float64)
    K = n.size
    L = block_layout(K)
    out = np.zeros(4 * K + 2)
    out[L["g"]] = g
    out[L["Hww"]] = H[0, 0]
    out[L["Hwb"]] = H[0, 1:]
    out[L["Hbb"]] = np.diag(H)[1:]
    out[L["n"]] = n
    return out


def dense_from_block(block) -> dict:
    """Inverse of block_from_dense: dict(g, H, n) with the arrow filled in."""
    block = np.asarray(block, np.float64)
    K = (block.size - 2) // 4
    L = block_layout(K)
    H = np.zeros((K + 1, K + 1))
    H[0, 0] = block[L["Hww"]][0]
    H[0, 1:] = H[1:, 0] = block[L["Hwb"]]
    H[np.arange(1, K + 1), np.arange(1, K + 1)] = block[L["Hbb"]]
    return dict(g=block[L["g"]].copy(), H=H, n=block[L["n"]].copy())


def sum_over_ranks_(block, group=None):
    """Sum `block` (a torch tensor) over the ranks of the default process
    group in place; a no-op without one or with a single rank."""
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(block, op=dist.ReduceOp.SUM, group=group)
    return block


def end_round(state, theta, damping_c: float = 10.0, group=None, stream=None):
    """End a refit round of a sharded batch: sum the AV state's accumulator
    block over the ranks, then solve on every rank (binding.AVState)."""
    sum_over_ranks_(state.accum(), group)
    state.solve(theta, damping_c, stream=stream)
