"""The allocation-free LM-head arg-max (head_argmax_noalloc).

Some callers cannot allocate device memory: code running where a framework's
allocator owns the device memory, or a serving loop that must not allocate
once started.  For them the library keeps the arg-max scratch in a fixed
device array of its own.  This test calls that entry point through the C ABI
and checks it against head_argmax with a caller-supplied workspace, on two
calls in a row (the shared array keeps the previous call's contents).  It sits
in a file collected last so that a run stopping at the first failure has run
every other test first.
"""
import numpy as np
import pytest

from q8_quantized_projection_gb300 import build, native, synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode,rows", [("i8", 16), ("f32", 3), ("f32", 8), ("i8x2", 1)])
def test_noalloc_head_matches_workspace_head(mode, rows):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    native.load()
    from oracle import oracle as orc
    orc.build()
    n, k = 20011, 1024
    q, s, h, pos = synth.planted_head(21 + rows, n, k, rows)
    x, _ = orc.rmsnorm(h)
    act = orc.quantize(mode, x)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda")
    qd, sd = dev(q), dev(s.view(np.int16))
    if mode == "f32":
        xq, xd = dev(act[0]), None
    elif mode == "i8":
        xq, xd = dev(act[0]), dev(act[1])
    else:
        xq, xd = dev(np.stack([act[0], act[1]])), dev(act[2])
    for call in range(2):
        tok_ref = torch.empty(rows, dtype=torch.int32, device="cuda")
        max_ref = torch.empty(rows, dtype=torch.float64, device="cuda")
        native.head_argmax(mode, qd, sd, xq, xd, rows, tok_ref, native.argmax_workspace(rows),
                           maxval=max_ref)
        tok = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
        mx = torch.empty(rows, dtype=torch.float64, device="cuda")
        native.head_argmax_noalloc(mode, qd, sd, xq, xd, rows, tok, maxval=mx)
        torch.cuda.synchronize()
        assert np.array_equal(tok.cpu().numpy(), tok_ref.cpu().numpy()), f"call {call}"
        assert np.array_equal(tok.cpu().numpy(), pos[np.arange(rows) % 8])
        rtol = 1e-9 if mode == "f32" else 1e-5
        assert np.allclose(mx.cpu().numpy(), max_ref.cpu().numpy(), rtol=rtol, atol=0)
    assert native.q8_device_error() == 0
