"""Tensor-parallel splits of the Q8_0 projection over the ranks of a process
group, one GPU per rank.

The pages split a layer over chips by its heads and FFN columns, each chip
holding its own slice of every projection, and sum the partial results of
the split the other way with an all-reduce, twice a layer (model::author,
Functions: check_tp, tp_decode_step, tp_decode_batch; spatial::streamed,
lower_tp_decode_streamed); the embedding and the head sit on the replicated
spine.  For the projection that gives two shardings and one reduction of the
head's arg-max:

* column split: rank r owns the contiguous output rows [n0, n1) of W (a
  multiple of the tensor-core tile where the rows allow); each rank projects
  its rows through the library, and an all-gather concatenates the outputs.
  Every output row is computed exactly as on one GPU.
* row split: rank r owns the K columns [k0, k1) of W, whole Q8_0 blocks, and
  the matching columns of the activation (codes and block scales are per
  block, so slicing at block boundaries keeps them); each rank projects its
  slice, and an all-reduce sums the partial outputs (f32, or f64 for the f32
  mode's f64 outputs).
* LM head: column split; each rank's arg-max over its rows, with its value,
  becomes a (value, global row) candidate, and an all-gather of the
  candidates ends in the library's own rule: the largest value, the lowest
  row on exact ties, NaN never the maximum, a head of NaN giving row 0.

Only host-side arithmetic on indices lives here (ranges and the choice among
candidates); every product runs in the library's kernels.  The local
projection is a parameter so that the host logic can also run without a GPU.
"""
from __future__ import annotations

import math

QK = 32
TILE_ROWS = 128   # weight rows of one tensor-core tile


def column_range(n: int, world: int, rank: int, align: int = TILE_ROWS):
    """Output rows [n0, n1) of rank `rank`: contiguous, disjoint, covering
    [0, n); boundaries on multiples of `align`, the ranks' shares of the
    aligned units as even as they divide."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank outside the group")
    units = -(-n // align)
    u0, u1 = units * rank // world, units * (rank + 1) // world
    return min(n, u0 * align), min(n, u1 * align)


def row_range(k: int, world: int, rank: int):
    """Reduction columns [k0, k1) of rank `rank`: whole 32-value blocks, as
    even as they divide."""
    if k % QK:
        raise ValueError("K must be a multiple of 32")
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank outside the group")
    nb = k // QK
    return QK * (nb * rank // world), QK * (nb * (rank + 1) // world)


def shard_columns(q, s, world: int, rank: int):
    """This rank's rows of a Q8_0 matrix (quants [N, K], scales [N, K/32])."""
    n0, n1 = column_range(q.shape[0], world, rank)
    return q[n0:n1], s[n0:n1], (n0, n1)


def shard_rows(q, s, world: int, rank: int):
    """This rank's reduction columns of a Q8_0 matrix, as contiguous arrays."""
    k0, k1 = row_range(q.shape[1], world, rank)
    qs = q[:, k0:k1]
    ss = s[:, k0 // QK:k1 // QK]
    qs = qs.contiguous() if hasattr(qs, "contiguous") else qs.copy()
    ss = ss.contiguous() if hasattr(ss, "contiguous") else ss.copy()
    return qs, ss, (k0, k1)


def slice_activation(mode: str, xq, xd, k0: int, k1: int):
    """The activation columns [k0, k1) in the library's layout: f32 [rows][K],
    one-word [rows][K] + scales [rows][K/32], two-word [2][rows][K] + scales."""
    def cont(a):
        return a.contiguous() if hasattr(a, "contiguous") else a.copy()
    if mode == "f32":
        return cont(xq[:, k0:k1]), None
    if mode == "i8":
        return cont(xq[:, k0:k1]), cont(xd[:, k0 // QK:k1 // QK])
    return cont(xq[:, :, k0:k1]), cont(xd[:, k0 // QK:k1 // QK])


def _native_proj(mode, q, s, xq, xd, rows, y):
    from q8_quantized_projection_gb300 import native
    native.q8_proj(mode, q, s, xq, xd, rows, y, out_f64=(y.dtype.itemsize == 8))


def _native_head(mode, q, s, xq, xd, rows):
    import torch
    from q8_quantized_projection_gb300 import native
    tok = torch.empty(rows, dtype=torch.int32, device=q.device)
    maxval = torch.empty(rows, dtype=torch.float64, device=q.device)
    native.head_argmax(mode, q, s, xq, xd, rows, tok, native.argmax_workspace(rows, device=q.device),
                       maxval=maxval)
    return tok, maxval


def tp_project_columns(mode, q_local, s_local, xq, xd, rows, n, group=None, proj=None,
                       out_dtype=None):
    """Column split: this rank's rows of W times the whole activation, then an
    all-gather; returns y [rows, n] on every rank."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    proj = proj or _native_proj
    dtype = out_dtype or torch.float32
    n0, n1 = column_range(n, world, rank)
    width = max(column_range(n, world, r)[1] - column_range(n, world, r)[0] for r in range(world))
    dev = q_local.device
    y_local = torch.zeros((rows, width), dtype=dtype, device=dev)
    if n1 > n0:
        part = torch.empty((rows, n1 - n0), dtype=dtype, device=dev)
        proj(mode, q_local, s_local, xq, xd, rows, part)
        y_local[:, :n1 - n0] = part
    gathered = [torch.empty_like(y_local) for _ in range(world)]
    dist.all_gather(gathered, y_local, group=group)
    pieces = []
    for r in range(world):
        a, b = column_range(n, world, r)
        pieces.append(gathered[r][:, :b - a])
    return torch.cat(pieces, dim=1)


def tp_project_rows(mode, q_local, s_local, xq_local, xd_local, rows, n, group=None, proj=None,
                    out_dtype=None):
    """Row split: this rank's reduction columns of W times the same columns of
    the activation (see slice_activation), then a sum over the ranks (an
    all-reduce); returns y [rows, n] on every rank."""
    import torch
    import torch.distributed as dist
    proj = proj or _native_proj
    dtype = out_dtype or torch.float32
    y = torch.empty((rows, n), dtype=dtype, device=q_local.device)
    proj(mode, q_local, s_local, xq_local, xd_local, rows, y)
    dist.all_reduce(y, op=dist.ReduceOp.SUM, group=group)
    return y


def combine_candidates(values, indices):
    """The arg-max over ranks of per-rank candidates (values [world][rows],
    global indices [world][rows], as lists or arrays): per row the largest
    value, the lowest index among equal values (-0 equal to +0), a NaN value
    no candidate; a row without any gives (0, NaN).  Returns (tokens, values)
    as lists."""
    world = len(values)
    rows = len(values[0]) if world else 0
    toks, vals = [], []
    for m in range(rows):
        bv, bi = None, None
        for r in range(world):
            v, i = float(values[r][m]), int(indices[r][m])
            if math.isnan(v):
                continue
            if bi is None or v > bv or (v == bv and i < bi):
                bv, bi = v, i
        if bi is None:
            toks.append(0)
            vals.append(float("nan"))
        else:
            toks.append(bi)
            vals.append(bv)
    return toks, vals


def tp_head_argmax(mode, q_local, s_local, xq, xd, rows, n, group=None, head=None):
    """LM head, column split: this rank's rows of the head and their arg-max,
    then the candidates of all ranks combined (combine_candidates); returns
    (tok int32 [rows], maxval float64 [rows]) on every rank."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    head = head or _native_head
    n0, n1 = column_range(n, world, rank)
    dev = q_local.device
    if n1 > n0:
        tok, val = head(mode, q_local, s_local, xq, xd, rows)
        cand = torch.stack([val.to(torch.float64), (tok.to(torch.float64) + n0)])
    else:   # no rows here: no candidate
        cand = torch.stack([torch.full((rows,), float("nan"), dtype=torch.float64, device=dev),
                            torch.zeros(rows, dtype=torch.float64, device=dev)])
    gathered = [torch.empty_like(cand) for _ in range(world)]
    dist.all_gather(gathered, cand, group=group)
    g = [x.cpu() for x in gathered]
    toks, vals = combine_candidates([x[0].tolist() for x in g], [x[1].tolist() for x in g])
    return (torch.tensor(toks, dtype=torch.int32, device=dev),
            torch.tensor(vals, dtype=torch.float64, device=dev))
