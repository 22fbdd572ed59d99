"""The batched oracle helper of the GPU tests (tests/moe_testlib.oracle_batch)
must give, token by token, what the oracle's per-token layer_decode gives:
same routing, weights and outputs to fp64 rounding.  CPU only."""
import numpy as np

from oracle import moe_oracle as O
from synth import generate as G
from tests.moe_testlib import oracle_batch


def test_oracle_batch_equals_per_token_layer_decode():
    H, I, E, K, B = 128, 64, 8, 3, 7
    ex = {e: G.expert(G.SEED, 5, e, H, I, 4) for e in range(E)}
    sh = G.expert(G.SEED, 5, G.SHARED_EXPERT, H, I, 2)
    R = G.router(G.SEED, 5, E, H)
    gamma = G.bf16_vector(G.SEED, 5, G.T_GAMMA, H, 1.0, 0.1)
    gate = G.bf16_vector(G.SEED, 5, G.T_SHARED_GATE, H, 0.0, 0.2)
    h = G.hidden_states(G.SEED, 5, B, H).astype(np.float64)
    off = np.stack([G.popularity_offsets(G.SEED, 5 + b, E) for b in range(B)])
    for shared, gate_bits in ((sh, gate), (sh, None), (None, None)):
        got = oracle_batch(h, experts=ex, shared=shared, router_bits=R, top_k=K, hidden=H, inter=I,
                           gamma_bits=gamma, shared_gate_bits=gate_bits, offset=off, threads=3)
        for b in range(B):
            ref = O.layer_decode(h[b], experts=ex, shared=shared, router_bits=R, top_k=K, hidden=H, inter=I,
                                 gamma_bits=gamma, shared_gate_bits=gate_bits, offset=off[b])
            assert list(got[b]["chosen"]) == list(ref["chosen"])
            assert np.allclose(got[b]["w"], ref["w"], rtol=0, atol=1e-15)
            assert np.allclose(got[b]["y"], ref["y"], rtol=1e-12, atol=1e-12)
            if shared is not None:
                assert got[b]["g_shared"] == ref["g_shared"]
