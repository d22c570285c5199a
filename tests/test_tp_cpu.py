"""The tensor-parallel splits (q8_quantized_projection_gb300.tp) on CPU:
the index arithmetic and the arg-max rule by hand, then world-size-2 gloo
ranks running the splits end to end with the CPU oracle standing in for the
library's local projection (the test's own injection; the library's path
passes its kernels), against the oracle's unsplit result."""
import math
import os
import socket
import sys

import numpy as np
import pytest

from q8_quantized_projection_gb300 import synth, tp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


# ------------------------------------------------------------ index arithmetic

@pytest.mark.parametrize("n", [1, 127, 128, 129, 4096, 6144, 28672, 128256, 1000])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_column_ranges_partition(n, world):
    ranges = [tp.column_range(n, world, r) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == n
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0 and a0 <= a1
    for a, b in ranges:
        assert a % tp.TILE_ROWS == 0 and (b % tp.TILE_ROWS == 0 or b == n)
    sizes = [b - a for a, b in ranges]
    # balanced to within one tile
    assert max(sizes) - min(sizes) <= tp.TILE_ROWS


@pytest.mark.parametrize("k", [32, 4096, 14336, 96])
@pytest.mark.parametrize("world", [1, 2, 4, 8])
def test_row_ranges_whole_blocks(k, world):
    ranges = [tp.row_range(k, world, r) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == k
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0
    assert all(a % 32 == 0 and b % 32 == 0 for a, b in ranges)
    with pytest.raises(ValueError):
        tp.row_range(k + 1, world, 0)


def test_combine_candidates_rule():
    nan, inf = float("nan"), float("inf")
    # per row: candidates of two ranks (value, global index)
    vals = [[3.0, 1.0, nan, -inf, -0.0, nan, 5.0],
            [3.0, 2.0, 4.0, -inf, 0.0, nan, 5.0]]
    idx = [[10, 10, 10, 10, 10, 10, 200],
           [200, 200, 200, 200, 200, 200, 100]]
    toks, best = tp.combine_candidates(vals, idx)
    assert toks == [10, 200, 200, 10, 10, 0, 100]
    assert best[:5] == [3.0, 2.0, 4.0, -inf, -0.0] and math.isnan(best[5]) and best[6] == 5.0


# ------------------------------------------------------------ gloo, 2 ranks

def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_act(mode, xq, xd):
    if mode == "f32":
        return (xq.numpy(),)
    if mode == "i8":
        return xq.numpy(), xd.numpy()
    return xq[0].numpy(), xq[1].numpy(), xd.numpy()


def _oracle_proj(mode, q, s, xq, xd, rows, y):
    import torch
    from oracle import oracle as orc
    yo, _ = orc.project(mode, q.numpy(), s.numpy().view(np.uint16), _oracle_act(mode, xq, xd))
    y.copy_(torch.from_numpy(np.ascontiguousarray(yo)).to(y.dtype))


def _oracle_head(mode, q, s, xq, xd, rows):
    import torch
    from oracle import oracle as orc
    tok, best, _ = orc.head_argmax(mode, q.numpy(), s.numpy().view(np.uint16), _oracle_act(mode, xq, xd))
    return torch.from_numpy(tok), torch.from_numpy(best.astype(np.float64))


def _inputs(mode, n, k, rows, seed):
    import torch
    from oracle import oracle as orc
    rng = np.random.default_rng(seed)
    q, s = synth.q8_weights(rng, n, k)
    x = synth.activations(rng, rows, k)
    act = orc.quantize(mode, orc.rmsnorm(x)[0])
    if mode == "f32":
        xq, xd = torch.from_numpy(act[0]), None
    elif mode == "i8":
        xq, xd = torch.from_numpy(act[0]), torch.from_numpy(act[1])
    else:
        xq, xd = torch.from_numpy(np.stack([act[0], act[1]])), torch.from_numpy(act[2])
    return q, s, act, xq, xd


# identical planted rows in pairs (rank 0 owns rows [0, 128) of 312)
TIE_PAIRS = [(127, 128), (200, 201), (3, 4), (0, 311), (50, 250), (126, 129), (100, 101),
             (260, 300)]


def _rank_main(rank, world, port, q_out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch
    import torch.distributed as dist
    from oracle import oracle as orc
    results = {}
    try:
        dist.init_process_group("gloo", rank=rank, world_size=world)
        for mode in ("f32", "i8", "i8x2"):
            n, k, rows = 300, 1024, 3
            qn, sn, act, xq, xd = _inputs(mode, n, k, rows, seed=5)
            y_full, norm = orc.project(mode, qn, sn, act)
            dt = torch.float64 if mode == "f32" else torch.float32
            qt, st = torch.from_numpy(qn), torch.from_numpy(sn.view(np.int16))
            # column split: every output row exactly as unsplit
            ql, sl, _ = tp.shard_columns(qt, st, world, rank)
            y = tp.tp_project_columns(mode, ql, sl, xq, xd, rows, n, proj=_oracle_proj, out_dtype=dt)
            col_ok = bool(np.array_equal(y.numpy().astype(np.float64), y_full.astype(np.float64)))
            # row split: partial sums over whole blocks, summed by the all-reduce
            qr, sr, (k0, k1) = tp.shard_rows(qt, st, world, rank)
            xqr, xdr = tp.slice_activation(mode, xq, xd, k0, k1)
            y2 = tp.tp_project_rows(mode, qr, sr, xqr, xdr, rows, n, proj=_oracle_proj, out_dtype=dt)
            err = np.abs(y2.numpy().astype(np.float64) - y_full.astype(np.float64))
            rtol = 1e-9 if mode == "f32" else 1e-5
            row_ok = bool(np.all(err <= rtol * norm + 1e-300))
            results[mode] = (col_ok, row_ok)
        # LM head: identical maximal rows (equal logits) in pairs, some on
        # both sides of the rank boundary at 128; the lower index must win
        n, k, rows = 312, 256, 16
        rng = np.random.default_rng(3)
        qh, sh = synth.q8_weights(rng, n, k)
        hh, base = synth.head_activations(rng, rows, k)
        for j, (p1, p2) in enumerate(TIE_PAIRS):
            synth.plant_head_rows(qh, sh, base[j:j + 1], np.array([p1]))
            qh[p2], sh[p2] = qh[p1], sh[p1]
        x_h, _ = orc.rmsnorm(hh)
        for mode in ("i8", "f32"):
            act = orc.quantize(mode, x_h)
            tok_full, best_full, _ = orc.head_argmax(mode, qh, sh, act)
            if mode == "f32":
                xq, xd = torch.from_numpy(act[0]), None
            else:
                xq, xd = torch.from_numpy(act[0]), torch.from_numpy(act[1])
            qt, st = torch.from_numpy(qh), torch.from_numpy(sh.view(np.int16))
            ql, sl, _ = tp.shard_columns(qt, st, world, rank)
            tok, val = tp.tp_head_argmax(mode, ql, sl, xq, xd, rows, n, head=_oracle_head)
            want = np.array([min(TIE_PAIRS[m % 8]) for m in range(rows)])
            results["head_" + mode] = (bool(np.array_equal(tok_full, want)),
                                       bool(np.array_equal(tok.numpy(), want)),
                                       bool(np.array_equal(val.numpy(), best_full.astype(np.float64))))
        q_out.put((rank, results))
    except Exception as e:  # reported to the parent, which fails the test
        import traceback
        q_out.put((rank, "error: " + repr(e) + traceback.format_exc()))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def test_two_rank_splits_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=300) for _ in procs]
    for p in procs:
        p.join(timeout=60)
    for rank, res in out:
        assert not isinstance(res, str), res
        for key, oks in res.items():
            assert all(oks), (rank, key, oks)
