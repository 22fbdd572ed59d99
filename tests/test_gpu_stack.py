"""Layer stack: tokens pass several layers in turn, h carried from layer to
layer, each layer with its own weights and its routing imposed by the reuse
trace through +30 logit offsets (the 40-layer workload's construction).

Through moe_layer_decode, one call per layer: each layer's output is checked
against the fp64 oracle run on that layer's input as the GPU saw it, and the
chosen experts must be the trace's.  Through moe_stack_decode, one call per
token (every layer in one launch of the single-token kernel): the routing of
every layer is the trace's, the token's output matches the oracle composed
over the layers, and the results equal those of the per-layer calls bit for
bit (the stack publishes each layer's fp32 output words unchanged, so its
arithmetic is the per-layer kernel's) -- also for stacks longer than one
launch, interleaved with single-layer calls on the same workspace (the epoch
and counter accounting), for the edge shapes, at full width, and after a
bounded wait ran out."""
import numpy as np
import pytest

from synth import generate as G
from tests.moe_testlib import REL_TOL, _to_dev, build_layer, pack_expert_device, rel_err, workspace

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_expert_matvec_moe_b300 as M  # noqa: E402

TINY = dict(hidden=256, inter=128, n_experts=16, top_k=4)
LAYERS, TOKENS = 3, 4


@pytest.fixture(scope="module", autouse=True)
def _build():
    from bit_expert_matvec_moe_b300 import build
    from synth import device

    build.build()
    device.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("path", ["fused", "multi"])
def test_layer_stack_follows_trace_and_matches_oracle(path):
    flags = M.MOE_HAS_SHARED | (M.MOE_NO_FUSED if path == "multi" else 0)
    dims = M.Dims(bits=4, flags=flags, **TINY)
    E, K = dims.n_experts, dims.top_k
    layers = [build_layer(dims, layer_id=l) for l in range(LAYERS)]
    trace = np.stack([G.reuse_trace(G.SEED, l, TOKENS, E, K) for l in range(LAYERS)])  # [L, T, K]
    h_all = G.hidden_states(G.SEED, 50, TOKENS, dims.hidden)
    ws = workspace(dims, 1)
    for t in range(TOKENS):
        h = torch.from_numpy(h_all[t:t + 1].copy()).cuda()
        for l, L in enumerate(layers):
            h_in = h.cpu().numpy()[0].astype(np.float64)
            off_np = G.trace_offsets(trace[l, t], E)
            off = torch.from_numpy(off_np[None, :].copy()).cuda()
            idx = torch.empty((1, K), dtype=torch.int32, device="cuda")
            M.moe_layer_decode(L.c_layer(), h, ws, logit_offset=off, idx_out=idx)
            assert M.moe_get_device_status(ws) == 0
            assert sorted(idx.cpu().numpy()[0].tolist()) == sorted(trace[l, t].tolist())
            ref = L.oracle(h_in, offset=off_np)
            y = h.cpu().numpy()[0]
            assert rel_err(y, ref["y"]) <= REL_TOL
            assert rel_err(y - h_in, ref["y"] - h_in) <= REL_TOL


# ----------------------------------------------------------------------------- moe_stack_decode
PATH_FLAGS = {"fused": 0, "fused_pdl": M.MOE_PDL, "multi": M.MOE_NO_FUSED}


def c_layer(L, flags_extra=0):
    d = L.dims
    if flags_extra:
        d = M.Dims(**{**d.__dict__, "flags": d.flags | flags_extra})
    return M.make_layer(d, L.experts, L.stride, L.router, shared=L.shared, shared_bits=L.shared_bits,
                        rms_gamma=L.gamma, shared_gate=L.gate)


def per_layer_calls(clayers, h_np, offs, ws):
    """The reference: one moe_layer_decode per layer on one token (each
    layer's offsets and outputs in buffers of their own: that call wants them
    16-byte aligned)."""
    d = clayers[0].d
    h = torch.from_numpy(np.ascontiguousarray(h_np, dtype=np.float32).reshape(1, -1)).cuda()
    idx = [torch.empty((1, d.top_k), dtype=torch.int32, device="cuda") for _ in clayers]
    w = [torch.empty((1, d.top_k), dtype=torch.float32, device="cuda") for _ in clayers]
    for l, c in enumerate(clayers):
        off = None if offs is None else offs[l:l + 1].clone()
        M.moe_layer_decode(c, h, ws, logit_offset=off, idx_out=idx[l], w_out=w[l])
    assert M.moe_get_device_status(ws) == 0
    return h.cpu().numpy()[0], torch.cat(idx).cpu().numpy(), torch.cat(w).cpu().numpy()


def stack_call(clayers, h_np, offs, ws):
    d = clayers[0].d
    h = torch.from_numpy(np.ascontiguousarray(h_np, dtype=np.float32).reshape(1, -1)).cuda()
    idx = torch.full((len(clayers), d.top_k), -1, dtype=torch.int32, device="cuda")
    w = torch.full((len(clayers), d.top_k), -1.0, dtype=torch.float32, device="cuda")
    M.moe_stack_decode(clayers, h, ws, logit_offset=offs, idx_out=idx, w_out=w)
    assert M.moe_get_device_status(ws) == 0
    return h.cpu().numpy()[0], idx.cpu().numpy(), w.cpu().numpy()


def trace_offsets(trace, t, E):
    """[L, E] offsets that impose token t's traced experts in every layer."""
    return torch.from_numpy(np.stack([G.trace_offsets(trace[l, t], E) for l in range(trace.shape[0])])).cuda()


@pytest.fixture(scope="module")
def tiny_layers():
    dims = M.Dims(bits=4, flags=M.MOE_HAS_SHARED, **TINY)
    return [build_layer(dims, layer_id=l) for l in range(LAYERS)]


@pytest.mark.parametrize("path", ["fused", "fused_pdl", "multi"])
def test_stack_call_follows_trace_and_matches_composed_oracle(tiny_layers, path):
    dims = tiny_layers[0].dims
    E, K = dims.n_experts, dims.top_k
    clayers = [c_layer(L, PATH_FLAGS[path]) for L in tiny_layers]
    trace = np.stack([G.reuse_trace(G.SEED, l, TOKENS, E, K) for l in range(LAYERS)])
    h_all = G.hidden_states(G.SEED, 51, TOKENS, dims.hidden)
    ws = workspace(dims, 1)
    for t in range(TOKENS):
        offs = trace_offsets(trace, t, E)
        y, idx, w = stack_call(clayers, h_all[t], offs, ws)
        offs_np = offs.cpu().numpy()
        ref = h_all[t].astype(np.float64)
        for l, L in enumerate(tiny_layers):
            assert sorted(idx[l].tolist()) == sorted(trace[l, t].tolist())
            out = L.oracle(ref, offset=offs_np[l])
            assert abs(float(w[l].sum()) - 1.0) < 1e-5
            ref = out["y"]
        assert rel_err(y, ref) <= REL_TOL
        assert rel_err(y - h_all[t], ref - h_all[t]) <= REL_TOL


EDGE = ["plain", "gamma_gate", "no_shared", "e_equals_k", "k1", "odd_shape", "two_bit", "two_bit_routed"]


def edge_layers(variant, n=3):
    shape, flags, bkw, bits = dict(TINY), M.MOE_HAS_SHARED, {}, 4
    if variant == "gamma_gate":
        flags |= M.MOE_HAS_SHARED_GATE
        bkw = dict(gamma=True, shared_gate=True)
    elif variant == "no_shared":
        flags = 0
    elif variant == "e_equals_k":
        shape.update(n_experts=4, top_k=4)
    elif variant == "k1":
        shape.update(top_k=1)
    elif variant == "odd_shape":
        shape = dict(hidden=320, inter=64, n_experts=24, top_k=3)
    elif variant == "two_bit":
        bits, bkw = 2, dict(shared_bits=2)
    elif variant == "two_bit_routed":
        bits = 2
    dims = M.Dims(bits=bits, flags=flags, **shape)
    return [build_layer(dims, layer_id=10 + l, **bkw) for l in range(n)]


@pytest.mark.parametrize("pdl", [False, True])
@pytest.mark.parametrize("variant", EDGE)
def test_stack_bitwise_equals_layer_calls(variant, pdl):
    layers = edge_layers(variant)
    dims = layers[0].dims
    clayers = [c_layer(L, M.MOE_PDL if pdl else 0) for L in layers]
    h_all = G.hidden_states(G.SEED, 52, 3, dims.hidden)
    ws_ref, ws = workspace(dims, 1), workspace(dims, 1)
    for t in range(3):
        offs = None if t == 0 else torch.from_numpy(
            G.hidden_states(G.SEED, 60 + t, len(layers), dims.n_experts)).cuda()  # arbitrary logit offsets
        y0, i0, w0 = per_layer_calls(clayers, h_all[t], offs, ws_ref)
        y1, i1, w1 = stack_call(clayers, h_all[t], offs, ws)
        assert np.array_equal(i0, i1) and np.array_equal(w0, w1)
        assert np.array_equal(y0, y1), float(np.max(np.abs(y0 - y1)))
    # one layer: the stack is the layer call
    y0, i0, w0 = per_layer_calls(clayers[:1], h_all[0], None, ws_ref)
    y1, i1, w1 = stack_call(clayers[:1], h_all[0], None, ws)
    assert np.array_equal(y0, y1) and np.array_equal(i0, i1) and np.array_equal(w0, w1)


def test_stack_longer_than_one_launch_and_interleaved(tiny_layers):
    """69 layers (64 in the first launch, 5 in the second), then single-layer
    calls and stacks of other lengths on the same workspace: every launch
    finds its epochs, results equal the per-layer calls."""
    clayers = [c_layer(L) for L in tiny_layers] * 23
    dims = tiny_layers[0].dims
    h_all = G.hidden_states(G.SEED, 53, 4, dims.hidden)
    ws_ref, ws = workspace(dims, 1), workspace(dims, 1)
    y0, i0, w0 = per_layer_calls(clayers, h_all[0], None, ws_ref)
    y1, i1, w1 = stack_call(clayers, h_all[0], None, ws)
    assert np.array_equal(y0, y1) and np.array_equal(i0, i1) and np.array_equal(w0, w1)
    for t, n in ((1, 1), (2, 2), (3, 7)):
        ya, _, _ = per_layer_calls(clayers[:n], h_all[t], None, ws)   # single-layer calls on the stack's workspace
        yb, _, _ = stack_call(clayers[:n], h_all[t], None, ws)
        yc, _, _ = per_layer_calls(clayers[:n], h_all[t], None, ws_ref)
        assert np.array_equal(ya, yc) and np.array_equal(yb, yc)


def test_stack_timeout_is_reported_and_recoverable(tiny_layers):
    """Every cross-block wait of the launch expects a later epoch (the
    workspace test hook): the blocks give up after their bounded waits, the
    status says TIMEOUT, and after the status is read the next stack call on the
    workspace gives the per-layer calls' result."""
    clayers = [c_layer(L) for L in tiny_layers]
    dims = tiny_layers[0].dims
    h_all = G.hidden_states(G.SEED, 54, 1, dims.hidden)
    ws = workspace(dims, 1)
    ws[:256].view(torch.int32)[4] = 1  # bar_extra
    h = torch.from_numpy(h_all.copy()).cuda()
    M.moe_stack_decode(clayers, h, ws)
    torch.cuda.synchronize()
    assert M.moe_get_device_status(ws) == 4  # MOE_ERR_TIMEOUT; header reset
    y1, i1, w1 = stack_call(clayers, h_all[0], None, ws)
    y0, i0, w0 = per_layer_calls(clayers, h_all[0], None, workspace(dims, 1))
    assert np.array_equal(y0, y1) and np.array_equal(i0, i1) and np.array_equal(w0, w1)


@pytest.mark.parametrize("pdl", [False, True])
def test_stack_full_width_bitwise_equals_layer_calls(pdl):
    """Four full-width layers (hidden 4096, 512 experts): one expert pool, and
    per layer its own router, shared expert and RMSNorm gamma, so that each
    layer's prefetched router and shared rows come from other addresses."""
    from synth import device as SD

    FULL = dict(hidden=4096, inter=1024, n_experts=512, top_k=4)
    flags = M.MOE_HAS_SHARED | (M.MOE_PDL if pdl else 0)
    dims = M.Dims(bits=4, flags=flags, **FULL)
    H, I, E = dims.hidden, dims.inter, dims.n_experts
    base = build_layer(M.Dims(bits=4, flags=M.MOE_HAS_SHARED, **FULL), gen="device")
    keep, clayers = [], []
    for l in range(4):
        router = _to_dev(G.router(G.SEED, 200 + l, E, H), torch, torch.int16)
        shared = torch.empty(M.moe_packed_expert_bytes(dims, 4), dtype=torch.uint8, device="cuda")
        pack_expert_device(dims, 4, SD.expert(G.SEED, 200 + l, G.SHARED_EXPERT, H, I, 4), shared, torch)
        gamma = _to_dev(G.bf16_vector(G.SEED, 200 + l, G.T_GAMMA, H, 1.0, 0.1), torch, torch.int16)
        keep += [router, shared, gamma]
        clayers.append(M.make_layer(dims, base.experts, base.stride, router, shared=shared, shared_bits=4,
                                    rms_gamma=gamma))
    torch.cuda.synchronize()
    h_all = G.hidden_states(G.SEED, 55, 3, H)
    ws_ref, ws = workspace(dims, 1), workspace(dims, 1)
    for t in range(3):
        y0, i0, w0 = per_layer_calls(clayers, h_all[t], None, ws_ref)
        y1, i1, w1 = stack_call(clayers, h_all[t], None, ws)
        assert np.array_equal(i0, i1) and np.array_equal(w0, w1)
        assert np.array_equal(y0, y1), float(np.max(np.abs(y0 - y1)))
