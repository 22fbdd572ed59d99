"""Layer stack: tokens pass several layers in turn through moe_layer_decode,
h updated in place and carried from layer to layer, each layer with its own
weights and its routing imposed by the reuse trace through +30 logit offsets
(the 40-layer workload's construction).  Each layer's output is checked
against the fp64 oracle run on that layer's input as the GPU saw it, and the
chosen experts must be the trace's."""
import numpy as np
import pytest

from synth import generate as G
from tests.moe_testlib import REL_TOL, build_layer, rel_err, workspace

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
