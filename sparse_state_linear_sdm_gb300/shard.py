"""Splitting one SDM forward pass over several GPUs (one process per GPU).

The (sequence, head) scans are independent, and so are the d_v columns of one table once
the slots are chosen ("Meccanismo Core" items 1, 3 and 4 of the Sparse Delta Memory
technical summary, gist.science/it/paper/2607.07386: the write and the read act on every
column of a selected row alike).  Two splits follow:

- by batch rows (weak scaling): rank r runs sequences r*B .. r*B + B - 1 on its own,
  with no collective at all (``batch_rows``); this is what the benchmark runs;
- by d_v columns (strong scaling of one batch): every rank runs the same selection
  (cheap, replicated), the planning pass and the scan on its contiguous slice of columns
  of the state and of v, and the output slices are gathered along d_v
  (``forward_dv_split``, one all-gather per pass).  A rank's slice of the state never
  leaves its GPU.

The per-rank work goes through the C ABI; the collective is torch.distributed's
all-gather (NCCL on GPUs), called on whole output tensors.  No kernel reads another GPU's
memory.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import api


def batch_rows(rank: int, B: int) -> tuple[int, int]:
    """Batch rows [r*B, (r+1)*B) of the logical workload that rank r runs (weak scaling)."""
    return rank * B, (rank + 1) * B


def dv_columns(d_v: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous column range [c0, c1) of d_v that rank `rank` of `world` owns.

    Every range has the same width, a multiple of 4 (the scan's 16-byte row pieces);
    d_v must be a multiple of 4 * world."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank or world size")
    if d_v % (4 * world):
        raise ValueError(f"d_v = {d_v} does not split into {world} slices of a multiple of 4 columns")
    w = d_v // world
    return rank * w, (rank + 1) * w


def _slice_cols(d_v: int, d_loc: int, B: int, H: int, W: int, R: int) -> int:
    """Columns per scan block for a slice: the full-width scan's choice when it divides the
    slice, so every column is computed by the same block arithmetic as without the split
    (bit-identical outputs); else the automatic choice for the slice."""
    full = api.scan_launch_info(B, H, d_v, W, R)["cols_per_cta"]
    return full if d_loc % full == 0 else 0


def scan_dv_slice(M0, sel, v, alpha, beta, rank: int, world: int, M_loc=None, workspace=None,
                  dev_err=None):
    """One rank's part of a d_v-split pass: the state slice M_loc [B, H, N, c1 - c0] started
    from M0[..., c0:c1] (M0=None: continue from M_loc) and the scan over the slice with the
    (replicated) selection `sel`.  Returns (o_loc [B, H, T, c1 - c0], M_loc)."""
    idx_w = sel[0]
    B, H, T, W = idx_w.shape
    R = sel[2].shape[3]
    d_v = v.shape[-1]
    c0, c1 = dv_columns(d_v, world, rank)
    if M_loc is None:
        if M0 is None:
            raise ValueError("M0=None continues from M_loc, which must then be given")
        N = M0.shape[1]
        M_loc = torch.empty((B, H, N, c1 - c0), dtype=torch.float32, device=v.device)
    if M0 is not None:
        api.init_state_from_M0(M_loc, M0[..., c0:c1].contiguous())
    o_loc = api.scan_forward(M_loc, *sel, v[..., c0:c1].contiguous(), alpha, beta, workspace=workspace,
                             dev_err=dev_err, cols_per_cta=_slice_cols(d_v, c1 - c0, B, H, W, R))
    return o_loc, M_loc


def gather_dv(o_loc: torch.Tensor, group=None) -> torch.Tensor:
    """All ranks' output slices, concatenated along d_v in rank order (one all-gather)."""
    world = dist.get_world_size(group)
    parts = [torch.empty_like(o_loc) for _ in range(world)]
    dist.all_gather(parts, o_loc.contiguous(), group=group)
    return torch.cat(parts, dim=-1)


def forward_dv_split(kp, qp, v, alpha, beta, M0, W: int, R: int, M_loc=None, group=None, dev_err=None):
    """One forward pass of a batch split over the ranks of `group` by d_v columns: the
    selection on every rank, the scan on this rank's column slice, then the all-gather of
    o.  Returns (o [B, H, T, d_v], M_loc, sel)."""
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    sel = api.select(kp, qp, W, R)
    o_loc, M_loc = scan_dv_slice(M0, sel, v, alpha, beta, rank, world, M_loc=M_loc, dev_err=dev_err)
    return gather_dv(o_loc, group), M_loc, sel
