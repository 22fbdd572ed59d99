"""Shared helpers of the GPU tests: build layers on the device from the seeded
generator, run the oracle on the same canonical arrays, compare."""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from oracle import moe_oracle as O
from synth import generate as G

# Tolerance of every floating-point parity check (the workload's bound):
# max_i |y_i - y*_i| / max(|y*_i|, FLOOR * max_j |y*_j|) <= REL_TOL
REL_TOL = 2e-3
FLOOR = 1e-3
TIE_EPS = 1e-6  # oracle logits closer than this may be chosen either way


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.maximum(np.abs(ref), FLOOR * np.max(np.abs(ref)))
    den = np.where(den == 0, 1.0, den)
    return float(np.max(np.abs(got - ref) / den))


def routing_ok(gpu_idx, logits64, k) -> tuple[bool, bool]:
    """(matches, tie): gpu_idx must equal the oracle's top-k, except that
    experts whose oracle logits are within TIE_EPS of the k-th may swap."""
    want = O.topk(logits64, k)
    if list(gpu_idx) == list(want):
        return True, False
    kth = logits64[want[-1]]
    near = set(np.nonzero(np.abs(logits64 - kth) < TIE_EPS)[0].tolist())
    sure = [e for e in want if e not in near]
    ok = all(e in gpu_idx for e in sure) and all((e in near) for e in gpu_idx if e not in want)
    ok = ok and len(set(gpu_idx.tolist())) == k
    return ok, True


@dataclass
class DeviceLayer:
    dims: object
    bits: int
    shared_bits: int
    seed: int
    layer_id: int
    experts: object = None  # torch uint8 [E, stride]
    stride: int = 0
    shared: object = None
    router: object = None   # torch int16 [E, H]
    router_np: object = None
    gamma: object = None
    gamma_np: object = None
    gate: object = None
    gate_np: object = None
    _cache: dict = field(default_factory=dict)

    def host_expert(self, e: int) -> dict:
        if e not in self._cache:
            H, I = self.dims.hidden, self.dims.inter
            if e == G.SHARED_EXPERT:
                self._cache[e] = G.expert(self.seed, self.layer_id, e, H, I, self.shared_bits)
            else:
                self._cache[e] = G.expert(self.seed, self.layer_id, e, H, I, self.bits)
        return self._cache[e]

    def c_layer(self):
        import bit_expert_matvec_moe_b300 as M

        return M.make_layer(self.dims, self.experts, self.stride, self.router, shared=self.shared,
                            shared_bits=self.shared_bits, rms_gamma=self.gamma, shared_gate=self.gate)

    def oracle_many(self, h, offset=None, threads: int = 8) -> list:
        """The oracle on every token of a batch (see oracle_batch)."""
        d = self.dims
        return oracle_batch(np.asarray(h, dtype=np.float64), experts=self.host_expert,
                            shared=self.host_expert(G.SHARED_EXPERT) if self.shared is not None else None,
                            router_bits=self.router_np, top_k=d.top_k, hidden=d.hidden, inter=d.inter,
                            eps=d.rms_eps, gamma_bits=self.gamma_np, shared_gate_bits=self.gate_np,
                            offset=offset, threads=threads)

    def oracle(self, h, offset=None, force_chosen=None) -> dict:
        d = self.dims
        return O.layer_decode(np.asarray(h, dtype=np.float64), experts=self.host_expert,
                              shared=self.host_expert(G.SHARED_EXPERT) if self.shared is not None else None,
                              router_bits=self.router_np, top_k=d.top_k, hidden=d.hidden, inter=d.inter,
                              eps=d.rms_eps, gamma_bits=self.gamma_np, shared_gate_bits=self.gate_np,
                              offset=offset, force_chosen=force_chosen)


def oracle_batch(h, *, experts, shared, router_bits, top_k, hidden, inter, eps=1e-6, gamma_bits=None,
                 shared_gate_bits=None, offset=None, threads: int = 8) -> list:
    """O.layer_decode on every row of h [B, H], composed from the oracle's own
    functions so that each touched expert is dequantised once: the routing of
    each token as in O.layer_decode, then O.expert_forward of each unique
    expert on the matrix whose columns are its tokens' xn (a matrix product is
    the matvec of each column), then the same combine.  Per token the result is
    the oracle's (tests/test_oracle_batch.py checks it against O.layer_decode).
    Experts are evaluated on a thread pool (numpy releases the GIL)."""
    from concurrent.futures import ThreadPoolExecutor

    get = experts if callable(experts) else (lambda e: experts[e])
    h = np.asarray(h, dtype=np.float64)
    B = h.shape[0]
    toks = []
    for b in range(B):
        xn = O.rmsnorm(h[b], gamma_bits, eps)
        logits = O.router_logits(router_bits, xn, None if offset is None else offset[b])
        chosen = O.topk(logits, top_k)
        toks.append({"xn": xn, "logits": logits, "chosen": chosen, "w": O.routing_weights(logits, chosen)})
    users = {}
    for b, t in enumerate(toks):
        for k, e in enumerate(t["chosen"]):
            users.setdefault(int(e), []).append((b, k))
    XN = np.stack([t["xn"] for t in toks], axis=1)  # [H, B]

    def run(item):
        e, lst = item
        cols = [b for b, _ in lst]
        return e, O.expert_forward(get(e), XN[:, cols], hidden, inter)["d"]

    with ThreadPoolExecutor(max_workers=max(1, threads)) as pool:
        d_by_e = dict(pool.map(run, sorted(users.items())))
        d_s = pool.submit(lambda: O.expert_forward(shared, XN, hidden, inter)["d"]).result() if shared is not None else None
    out = []
    for b, t in enumerate(toks):
        d_routed = []
        for k, e in enumerate(t["chosen"]):
            col = [bb for bb, _ in users[int(e)]].index(b)
            d_routed.append(d_by_e[int(e)][:, col])
        y = h[b].copy()
        for wk, dk in zip(t["w"], d_routed):
            y = y + wk * dk
        r = {**t, "d_routed": d_routed}
        if shared is not None:
            g_s = 1.0
            if shared_gate_bits is not None:
                g_s = 1.0 / (1.0 + np.exp(-(O.bf16_to_f64(shared_gate_bits) @ t["xn"])))
            y = y + g_s * d_s[:, b]
            r["d_shared"] = d_s[:, b]
            r["g_shared"] = g_s
        r["y"] = y
        out.append(r)
    return out


def _to_dev(arr, torch, dtype=None):
    a = np.ascontiguousarray(arr)
    if dtype is not None and a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def pack_expert_device(dims, bits, canon, dst, torch):
    """canon: dict with gate/up/down (codes, scales, biases) as numpy or torch."""
    import bit_expert_matvec_moe_b300 as M

    codes, scales, biases = [], [], []
    for m in ("gate", "up", "down"):
        c, s, b = canon[m]
        if isinstance(c, np.ndarray):
            c = _to_dev(c, torch)
            s = _to_dev(s, torch, torch.int16)
            b = _to_dev(b, torch, torch.int16)
        codes.append(c)
        scales.append(s)
        biases.append(b)
    M.moe_pack_weights(dims, bits, codes, scales, biases, dst)


def build_layer(dims, seed=G.SEED, layer_id=0, shared_bits=4, gen="host", gamma=False, shared_gate=False,
                stride_pad=0) -> DeviceLayer:
    """Generate, upload and pack one layer.  gen='device' uses the CUDA twin of
    the generator (bit-identical to the host one) for the expert weights."""
    import torch

    import bit_expert_matvec_moe_b300 as M
    from synth import device as SD

    H, I, E = dims.hidden, dims.inter, dims.n_experts
    L = DeviceLayer(dims=dims, bits=dims.bits, shared_bits=shared_bits, seed=seed, layer_id=layer_id)
    blob = M.moe_packed_expert_bytes(dims, dims.bits)
    L.stride = blob + stride_pad
    L.experts = torch.empty((E, L.stride), dtype=torch.uint8, device="cuda")
    for e in range(E):
        canon = SD.expert(seed, layer_id, e, H, I, dims.bits) if gen == "device" else G.expert(seed, layer_id, e, H, I, dims.bits)
        pack_expert_device(dims, dims.bits, canon, L.experts[e], torch)
    if dims.flags & M.MOE_HAS_SHARED:
        L.shared = torch.empty(M.moe_packed_expert_bytes(dims, shared_bits), dtype=torch.uint8, device="cuda")
        canon = (SD.expert(seed, layer_id, G.SHARED_EXPERT, H, I, shared_bits) if gen == "device"
                 else G.expert(seed, layer_id, G.SHARED_EXPERT, H, I, shared_bits))
        pack_expert_device(dims, shared_bits, canon, L.shared, torch)
    L.router_np = G.router(seed, layer_id, E, H)
    L.router = _to_dev(L.router_np, torch, torch.int16)
    if gamma:
        L.gamma_np = G.bf16_vector(seed, layer_id, G.T_GAMMA, H, 1.0, 0.1)
        L.gamma = _to_dev(L.gamma_np, torch, torch.int16)
    if shared_gate:
        L.gate_np = G.bf16_vector(seed, layer_id, G.T_SHARED_GATE, H, 0.0, 0.02)
        L.gate = _to_dev(L.gate_np, torch, torch.int16)
    torch.cuda.synchronize()
    return L


def workspace(dims, max_batch):
    import torch

    import bit_expert_matvec_moe_b300 as M

    n = M.moe_workspace_bytes(dims, max_batch)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    M.moe_workspace_init(ws)
    return ws
