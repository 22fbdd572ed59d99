"""moe_layer_decode_noalloc: the single-token layer for callers that cannot
allocate device memory (they are handed their input and output buffers only,
e.g. inside another framework's memory pool or an allocation-free hot path).
It keeps its cross-block state in the library's fixed device array instead of
a caller workspace.  Its output must match moe_layer_decode's on the same
inputs, on consecutive calls (the array carries its state from call to call).
This file is collected last, so a failure here comes after every other test."""
import numpy as np
import pytest

from synth import generate as G
from tests.moe_testlib import REL_TOL, build_layer, rel_err, routing_ok, workspace

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_expert_matvec_moe_b300 as M  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _build():
    from bit_expert_matvec_moe_b300 import build
    from synth import device

    build.build()
    device.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _decode_with_workspace(L, h_np):
    h = torch.from_numpy(h_np.copy()).cuda()
    idx = torch.empty((1, L.dims.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((1, L.dims.top_k), dtype=torch.float32, device="cuda")
    ws = workspace(L.dims, 1)
    M.moe_layer_decode(L.c_layer(), h, ws, idx_out=idx, w_out=w)
    assert M.moe_get_device_status(ws) == 0
    return h.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


def _decode_noalloc(L, h_np):
    h = torch.from_numpy(h_np.copy()).cuda()
    idx = torch.empty((1, L.dims.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((1, L.dims.top_k), dtype=torch.float32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    M.moe_layer_decode_noalloc(L.c_layer(), h, status, idx_out=idx, w_out=w)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return h.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("shape", [dict(hidden=256, inter=128, n_experts=16, top_k=4),
                                   dict(hidden=4096, inter=1024, n_experts=64, top_k=4)])
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(shape):
    L = build_layer(M.Dims(flags=M.MOE_HAS_SHARED, **shape), gen="device" if shape["hidden"] > 1024 else "host")
    hs = G.hidden_states(G.SEED, 41, 2, shape["hidden"])
    for t in range(2):  # two calls in a row on the shared array
        y_ref, idx_ref, w_ref = _decode_with_workspace(L, hs[t:t + 1])
        y, idx, w = _decode_noalloc(L, hs[t:t + 1])
        assert np.array_equal(idx, idx_ref)
        assert rel_err(w, w_ref) <= REL_TOL
        assert rel_err(y[0], y_ref[0]) <= REL_TOL
        assert rel_err(y[0] - hs[t], y_ref[0] - hs[t]) <= REL_TOL
        # and against the oracle itself, not only the other CUDA entry point
        ref = L.oracle(hs[t])
        ok, tie = routing_ok(idx[0], ref["logits"], L.dims.top_k)
        assert ok
        if tie:
            ref = L.oracle(hs[t], force_chosen=idx[0])
        assert rel_err(y[0], ref["y"]) <= REL_TOL
        assert rel_err(y[0] - hs[t], ref["y"] - hs[t]) <= REL_TOL


def test_noalloc_rejects_layers_beyond_its_array():
    """A layer whose cross-block state exceeds the fixed array is refused with a
    clear error before anything is enqueued."""
    from bit_expert_matvec_moe_b300 import _native as N

    d = M.Dims(hidden=4096, inter=4096, n_experts=1024, top_k=8, flags=M.MOE_HAS_SHARED)
    stride = M.moe_packed_expert_bytes(d, 4)
    fake = torch.empty(16, dtype=torch.uint8, device="cuda")
    router = torch.empty((1024, 4096), dtype=torch.int16, device="cuda")
    layer = M.make_layer(d, fake, stride, router, shared=fake)
    h = torch.zeros((1, 4096), dtype=torch.float32, device="cuda")
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    with pytest.raises(M.MoeError) as err:
        M.moe_layer_decode_noalloc(layer, h, status)
    assert err.value.status == N.MOE_ERR_UNSUPPORTED
    assert "scratch array" in str(N.load().moe_last_error_message().decode())


def test_noalloc_requires_a_status_word():
    """The status copy is the only record of a device-side error (the array is
    out of the caller's reach and the next call clears it), so the C entry
    point refuses a NULL status pointer."""
    from bit_expert_matvec_moe_b300 import _native as N

    L = build_layer(M.Dims(flags=M.MOE_HAS_SHARED, hidden=256, inter=128, n_experts=16, top_k=4))
    h = torch.from_numpy(G.hidden_states(G.SEED, 42, 1, 256)).cuda()
    lib = N.load()
    layer = L.c_layer()
    import ctypes

    st = lib.moe_layer_decode_noalloc(ctypes.byref(layer), h.data_ptr(), None, None, None, None,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == N.MOE_ERR_INVALID_ARG


def test_noalloc_timeout_is_reported_then_the_next_call_recovers():
    """The path unique to this entry point: a bounded cross-block wait runs out
    (the library's one-shot test hook makes every wait of the launch expect a
    later launch's data; each block gives up after 1 s, no fault), status_out
    carries the timeout bit, and the next call - which clears the error state
    of the array itself - matches moe_layer_decode and the oracle."""
    from bit_expert_matvec_moe_b300 import _native as N

    L = build_layer(M.Dims(flags=M.MOE_HAS_SHARED, hidden=256, inter=128, n_experts=16, top_k=4))
    hs = G.hidden_states(G.SEED, 43, 2, 256)
    assert N.load().moe_noalloc_test_timeout_next() == 0
    h = torch.from_numpy(hs[0:1].copy()).cuda()
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    M.moe_layer_decode_noalloc(L.c_layer(), h, status)
    torch.cuda.synchronize()
    assert int(status.item()) & 1  # ST_TIMEOUT
    # the following call runs normally on the same array
    y_ref, idx_ref, w_ref = _decode_with_workspace(L, hs[1:2])
    y, idx, w = _decode_noalloc(L, hs[1:2])
    assert np.array_equal(idx, idx_ref)
    assert rel_err(w, w_ref) <= REL_TOL
    assert rel_err(y[0], y_ref[0]) <= REL_TOL
    ref = L.oracle(hs[1])
    ok, tie = routing_ok(idx[0], ref["logits"], L.dims.top_k)
    assert ok
    if tie:
        ref = L.oracle(hs[1], force_chosen=idx[0])
    assert rel_err(y[0], ref["y"]) <= REL_TOL
