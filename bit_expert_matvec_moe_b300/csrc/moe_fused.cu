// Fused single-token MoE layer: one cooperative launch of one block per SM.
//
// Block c of P owns gate/up row pairs [c*I/P, (c+1)*I/P) of every expert the
// token uses and down rows [c*H/P, (c+1)*H/P).  Its weight bytes arrive by
// bulk copies (TMA engine) into shared memory:
//   start        shared expert: gate/up rows (ring slot 0) and down rows
//   after top-K  routed experts: gate/up rows through a ring of staging slots,
//                all down rows at once (they are consumed last)
// Phases, with the two grid-wide waits the data dependencies require:
//   RMSNorm + activation limbs (redundant per block)
//   router rows c, c+P, ... -> logits (global)          -- arrive barrier 1
//   shared-expert gate/up + SwiGLU (already staged)
//   wait barrier 1; top-K of all logits (redundant per block, identical result)
//   routed gate/up + SwiGLU -> a (global)               -- barrier 2
//   limbs of every a; down rows of all experts, weighted combine + residual.
// Nothing returns to the host inside the layer; routing is read from shared
// memory by the block that issues the copies.  Every wait is bounded (1 s):
// on timeout the block records MOE_ERR_TIMEOUT, waits for its own copies in
// flight and leaves, and later launches on the same workspace return at once.
#include "moe_internal.h"

namespace moe {

namespace {

__device__ __forceinline__ size_t lo_row(int c, int P, int n) { return (size_t)c * n / P; }

template <int BITS>
__device__ __forceinline__ void gu_rows(const uint8_t* slot, const Fmt& f, int nr, const uint32_t* xq, const float2* xe,
                                        float* part, int wid, int lane) {
  auto off = [&](int r) { return (size_t)(r >> 1) * f.gu_pair + (size_t)(r & 1) * f.gu_row; };
  rows_dot<BITS>(slot, off, 2 * nr, f.ng_h, f.gu_codes, xq, xe, part, wid, kBlock / 32, lane);
}

template <int BITS>
__device__ __forceinline__ void dn_rows(const uint8_t* area, const Fmt& f, int nj, const uint32_t* aq, const float2* ae,
                                        float* part, int wid, int lane) {
  auto off = [&](int r) { return (size_t)r * f.d_row; };
  rows_dot<BITS>(area, off, nj, f.ng_i, f.d_codes, aq, ae, part, wid, kBlock / 32, lane);
}

}  // namespace

__global__ void __launch_bounds__(kBlock, 1) fused_decode_kernel(const FusedArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  const FusedPlan& pl = a.plan;
  float* xbuf = reinterpret_cast<float*>(sm + pl.off_x);  // xn, later the limbs of every a
  uint32_t* xq4 = reinterpret_cast<uint32_t*>(sm + pl.off_xq4);
  uint32_t* xq2 = reinterpret_cast<uint32_t*>(sm + pl.off_xq2);
  float2* xe4 = reinterpret_cast<float2*>(sm + pl.off_xe4);
  float2* xe2 = reinterpret_cast<float2*>(sm + pl.off_xe2);
  float2* ae = reinterpret_cast<float2*>(sm + pl.off_ae);
  float* part = reinterpret_cast<float*>(sm + pl.off_part);
  float* pd = reinterpret_cast<float*>(sm + pl.off_pd);
  float* slog = reinterpret_cast<float*>(sm + pl.off_logits);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + pl.off_bar);  // [nslots] gate/up, then [NE] down

  __shared__ float s_red[kBlock / 32];
  __shared__ float s_rpart[64];
  __shared__ unsigned long long s_cand[(kBlock / 32) * kMaxTopK];
  __shared__ int s_idx[kMaxTopK];
  __shared__ float s_w[kMaxTopK];
  __shared__ float s_coef[kMaxTopK + 1];
  __shared__ int s_flag, s_abort;
  __shared__ uint32_t s_gu_issued[kMaxSlots], s_gu_done[kMaxSlots], s_dn_issued, s_dn_done;

  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int P = gridDim.x, c = blockIdx.x;
  const int NE = a.K + a.has_shared;
  const Fmt fr = make_fmt(a.bits, a.H, a.I);
  const Fmt fs = make_fmt(a.shared_bits, a.H, a.I);
  const int r0 = (int)lo_row(c, P, a.I), nr = (int)lo_row(c + 1, P, a.I) - r0;
  const int j0 = (int)lo_row(c, P, a.H), nj = (int)lo_row(c + 1, P, a.H) - j0;
  const int ns = pl.nslots;
  uint64_t* gu_bar = bar;
  uint64_t* dn_bar = bar + ns;

  if (tid == 0) {
    for (int i = 0; i < ns + NE; ++i) mbar_init(&bar[i], 1);
    fence_mbar_init();
    for (int i = 0; i < kMaxSlots; ++i) s_gu_issued[i] = s_gu_done[i] = 0u;
    s_dn_issued = s_dn_done = 0u;
    s_abort = *(volatile uint32_t*)&a.hdr->abort ? 1 : 0;
  }
  __syncthreads();
  if (s_abort) return;

  // expert p (0 .. NE-1): p = 0 is the shared expert when present
  auto expert_blob = [&](int p) -> const uint8_t* {
    if (a.has_shared && p == 0) return a.shared;
    const int k = p - a.has_shared;
    return a.experts + (size_t)s_idx[k] * a.stride;
  };
  auto expert_fmt = [&](int p) -> const Fmt& { return (a.has_shared && p == 0) ? fs : fr; };
  // thread 0: stage expert p's gate/up rows into slot p % ns
  auto issue_gu = [&](int p) {
    const Fmt& f = expert_fmt(p);
    const int sl = p % ns;
    if (nr > 0) {
      const uint32_t bytes = (uint32_t)nr * f.gu_pair;
      mbar_expect_tx(&gu_bar[sl], bytes);
      bulk_g2s(sm + pl.off_gu + sl * pl.slot_bytes, expert_blob(p) + (size_t)r0 * f.gu_pair, bytes, &gu_bar[sl]);
      s_gu_issued[sl]++;
    }
  };
  auto issue_dn = [&](int p) {
    const Fmt& f = expert_fmt(p);
    if (nj > 0) {
      const uint32_t bytes = (uint32_t)nj * f.d_row;
      mbar_expect_tx(&dn_bar[p], bytes);
      bulk_g2s(sm + pl.off_dn[p], expert_blob(p) + f.d_off + (size_t)j0 * f.d_row, bytes, &dn_bar[p]);
      s_dn_issued |= 1u << p;
    }
  };
  // all threads: bounded wait for slot sl's next phase; false on timeout
  auto wait_gu = [&](int sl) -> bool {
    if (nr == 0) return true;
    const uint32_t ph = s_gu_done[sl] & 1u;
    const bool ok = mbar_wait(&gu_bar[sl], ph);
    if (!ok) s_abort = 1;
    __syncthreads();
    if (tid == 0 && !s_abort) s_gu_done[sl]++;
    __syncthreads();
    return !s_abort;
  };

  // ---- stage the shared expert before anything else
  if (tid == 0 && a.has_shared) {
    issue_gu(0);
    issue_dn(0);
  }

  // ---- RMSNorm (fixed-order reduction: identical in every block)
  float hres = 0.f;
  if (tid < nj) hres = a.h[j0 + tid];
  float ss = 0.f;
  for (int i = tid; i < a.H; i += kBlock) {
    const float x = a.h[i];
    xbuf[i] = x;
    ss = fmaf(x, x, ss);
  }
  ss = warp_sum(ss);
  if (lane == 0) s_red[wid] = ss;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int w = 0; w < kBlock / 32; ++w) t += s_red[w];
    s_red[0] = 1.0f / sqrtf(t / (float)a.H + a.eps);
  }
  __syncthreads();
  const float rs = s_red[0];
  for (int i = tid; i < a.H; i += kBlock) {
    float x = xbuf[i] * rs;
    if (a.gamma) x *= bf16lo(a.gamma[i]);
    xbuf[i] = x;
  }
  __syncthreads();

  // ---- activation limbs for the code widths in use
  const bool need4 = (a.bits == 4) || (a.has_shared && a.shared_bits == 4);
  const bool need2 = (a.bits == 2) || (a.has_shared && a.shared_bits == 2);
  bool finite = true;
  for (int g = wid; g < fr.ng_h; g += kBlock / 32) {
    const float x0 = xbuf[g * kGroup + 2 * lane], x1 = xbuf[g * kGroup + 2 * lane + 1];
    if (need4) finite &= quantize_group<4>(x0, x1, lane, reinterpret_cast<uint8_t*>(xq4 + g * kLimbWords), xe4 + g);
    if (need2) finite &= quantize_group<2>(x0, x1, lane, reinterpret_cast<uint8_t*>(xq2 + g * kLimbWords), xe2 + g);
  }
  const int nonfinite_x = __syncthreads_or(!finite);

  // ---- router rows e = c + P t (row E = shared-expert gate vector)
  {
    const int nrows_all = a.E + (a.has_gate ? 1 : 0);
    const int nmine = c < nrows_all ? (nrows_all - 1 - c) / P + 1 : 0;
    const int nq = (a.H % 1024 == 0 && nmine * 4 <= 64) ? 4 : 1;  // column quarters per row
    const int qlen = a.H / nq;
    for (int t = wid; t < nmine * nq; t += kBlock / 32) {
      const int ri = t / nq, q = t % nq;
      const int e = c + P * ri;
      const uint16_t* R = e < a.E ? a.router + (size_t)e * a.H : a.gate;
      float acc = 0.f;
      for (int col = q * qlen + 8 * lane; col < (q + 1) * qlen; col += 256) {
        const uint4 rw = __ldg(reinterpret_cast<const uint4*>(R + col));
        const float4 xa = *reinterpret_cast<const float4*>(xbuf + col);
        const float4 xb = *reinterpret_cast<const float4*>(xbuf + col + 4);
        acc = fmaf(bf16lo(rw.x), xa.x, acc); acc = fmaf(bf16hi(rw.x), xa.y, acc);
        acc = fmaf(bf16lo(rw.y), xa.z, acc); acc = fmaf(bf16hi(rw.y), xa.w, acc);
        acc = fmaf(bf16lo(rw.z), xb.x, acc); acc = fmaf(bf16hi(rw.z), xb.y, acc);
        acc = fmaf(bf16lo(rw.w), xb.z, acc); acc = fmaf(bf16hi(rw.w), xb.w, acc);
      }
      acc = warp_sum(acc);
      if (lane == 0) s_rpart[t] = acc;
    }
    __syncthreads();
    if (tid < nmine) {
      const int e = c + P * tid;
      float v = 0.f;
      for (int q = 0; q < nq; ++q) v += s_rpart[tid * nq + q];
      if (e < a.E && a.offset) v += a.offset[e];
      a.logits[e] = v;
      __threadfence();
    }
  }
  __syncthreads();
  uint32_t gen1 = 0;
  if (tid == 0) gen1 = grid_arrive(a.hdr, (uint32_t)P);

  // ---- shared expert gate/up while the other blocks finish routing
  if (a.has_shared) {
    if (!wait_gu(0)) goto cleanup;
    if (nr > 0) {
      if (a.shared_bits == 4)
        gu_rows<4>(sm + pl.off_gu, fs, nr, xq4, xe4, part, wid, lane);
      else
        gu_rows<2>(sm + pl.off_gu, fs, nr, xq2, xe2, part, wid, lane);
    }
    __syncthreads();
    if (tid < nr) {
      const RowMap m = make_rowmap(fs.ng_h);
      float g = 0.f, u = 0.f;
      for (int ch = 0; ch < m.chunks; ++ch) {
        g += part[(2 * tid) * m.chunks + ch];
        u += part[(2 * tid + 1) * m.chunks + ch];
      }
      a.a_glob[r0 + tid] = silu_mul(g, u);
    }
  }

  // ---- routing result
  if (tid == 0) {
    if (!grid_wait(a.hdr, gen1)) s_abort = 1;
  }
  __syncthreads();
  if (s_abort) goto cleanup;
  for (int e = tid; e < a.E + (a.has_gate ? 1 : 0); e += kBlock) slog[e] = __ldcg(a.logits + e);
  __syncthreads();
  {
    const bool ok = block_topk(slog, a.E, a.K, s_cand, s_idx, s_w, &s_flag);
    if (tid == 0) {
      for (int k = 0; k < a.K; ++k) s_coef[a.has_shared + k] = s_w[k];
      if (a.has_shared) s_coef[0] = a.has_gate ? 1.0f / (1.0f + expf(-slog[a.E])) : 1.0f;
      if (c == 0) {
        if (!ok || nonfinite_x) atomicOr(&a.hdr->status, ST_NONFINITE);
        for (int k = 0; k < a.K; ++k) {
          if (a.idx_out) a.idx_out[k] = s_idx[k];
          if (a.w_out) a.w_out[k] = s_w[k];
        }
      }
      // routed gate/up copies into free slots, then every routed down block
      fence_proxy_async();
      for (int p = a.has_shared; p < NE && p < a.has_shared + ns; ++p) issue_gu(p);
      for (int p = a.has_shared; p < NE; ++p) issue_dn(p);
    }
    __syncthreads();
  }

  // ---- routed gate/up + SwiGLU
  for (int p = a.has_shared; p < NE; ++p) {
    const int sl = p % ns;
    if (!wait_gu(sl)) goto cleanup;
    const uint8_t* slot = sm + pl.off_gu + sl * pl.slot_bytes;
    if (nr > 0) {
      if (a.bits == 4)
        gu_rows<4>(slot, fr, nr, xq4, xe4, part, wid, lane);
      else
        gu_rows<2>(slot, fr, nr, xq2, xe2, part, wid, lane);
    }
    __syncthreads();
    if (tid < nr) {
      const RowMap m = make_rowmap(fr.ng_h);
      float g = 0.f, u = 0.f;
      for (int ch = 0; ch < m.chunks; ++ch) {
        g += part[(2 * tid) * m.chunks + ch];
        u += part[(2 * tid + 1) * m.chunks + ch];
      }
      a.a_glob[(size_t)p * a.I + r0 + tid] = silu_mul(g, u);
    }
    if (tid == 0 && p + ns < NE) {
      fence_proxy_async();
      issue_gu(p + ns);
    }
    __syncthreads();
  }

  // ---- every a complete
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t g2 = grid_arrive(a.hdr, (uint32_t)P);
    if (!grid_wait(a.hdr, g2)) s_abort = 1;
  }
  __syncthreads();
  if (s_abort) goto cleanup;

  // ---- limbs of a for each expert (layout of that expert's code width)
  {
    uint32_t* aq = reinterpret_cast<uint32_t*>(xbuf);
    for (int t = wid; t < NE * fr.ng_i; t += kBlock / 32) {
      const int p = t / fr.ng_i, g = t % fr.ng_i;
      const float* av = a.a_glob + (size_t)p * a.I + g * kGroup;
      const float x0 = __ldcg(av + 2 * lane), x1 = __ldcg(av + 2 * lane + 1);
      uint8_t* q = reinterpret_cast<uint8_t*>(aq + (size_t)t * kLimbWords);
      if (expert_fmt(p).bits == 4)
        quantize_group<4>(x0, x1, lane, q, ae + t);
      else
        quantize_group<2>(x0, x1, lane, q, ae + t);
    }
    __syncthreads();

    // ---- down rows of every expert, then combine + residual
    for (int p = 0; p < NE; ++p) {
      if (nj > 0) {
        const bool ok = mbar_wait(&dn_bar[p], 0);
        if (!ok) s_abort = 1;
        __syncthreads();
        if (s_abort) goto cleanup;
        if (tid == 0) s_dn_done |= 1u << p;
        const Fmt& f = expert_fmt(p);
        const RowMap m = make_rowmap(f.ng_i);
        float* pp = pd + (size_t)p * pl.rows_d * m.chunks;
        const uint32_t* q = aq + (size_t)p * fr.ng_i * kLimbWords;
        if (f.bits == 4)
          dn_rows<4>(sm + pl.off_dn[p], f, nj, q, ae + p * fr.ng_i, pp, wid, lane);
        else
          dn_rows<2>(sm + pl.off_dn[p], f, nj, q, ae + p * fr.ng_i, pp, wid, lane);
      }
    }
    __syncthreads();
    if (tid < nj) {
      float y = 0.f;
      for (int p = 0; p < NE; ++p) {
        const RowMap m = make_rowmap(expert_fmt(p).ng_i);
        const float* pp = pd + (size_t)p * pl.rows_d * m.chunks;
        float d = 0.f;
        for (int ch = 0; ch < m.chunks; ++ch) d += pp[tid * m.chunks + ch];
        y = fmaf(s_coef[p], d, y);
      }
      a.h[j0 + tid] = hres + y;
    }
  }
  return;

cleanup:
  // leave only after this block's own copies in flight have landed
  __syncthreads();
  if (tid == 0) {
    for (int sl = 0; sl < ns; ++sl)
      if (s_gu_issued[sl] > s_gu_done[sl]) mbar_wait(&gu_bar[sl], s_gu_done[sl] & 1u);
    for (int p = 0; p < NE; ++p)
      if ((s_dn_issued >> p & 1u) && !(s_dn_done >> p & 1u)) mbar_wait(&dn_bar[p], 0);
  }
  __syncthreads();
}

bool fused_plan(int H, int I, int E, int K, int bits, int shared_bits, int has_shared, int device, FusedPlan* out) {
  int nsm = 0, optin = 0;
  if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess) return false;
  const int NE = K + has_shared;
  const Fmt fr = make_fmt(bits, H, I);
  const Fmt fs = make_fmt(has_shared ? shared_bits : bits, H, I);
  FusedPlan p{};
  p.P = nsm;
  p.rows_gu = (I + nsm - 1) / nsm;
  p.rows_d = (H + nsm - 1) / nsm;
  p.slot_bytes = pad16((size_t)p.rows_gu * std::max(fr.gu_pair, fs.gu_pair));
  const RowMap mh = make_rowmap(fr.ng_h), mi = make_rowmap(fr.ng_i);
  if (mh.chunks > kBlock / 32 || mi.chunks > kBlock / 32) return false;
  if ((E + 1 + nsm - 1) / nsm > 64) return false;  // router partials per block
  const bool need4 = bits == 4 || (has_shared && shared_bits == 4);
  const bool need2 = bits == 2 || (has_shared && shared_bits == 2);
  // static shared memory of the kernel is small; keep 4 KB of headroom for it
  const size_t budget = (size_t)optin - 4096;
  for (int ns = kMaxSlots; ns >= 2; --ns) {
    size_t o = 0;
    auto take = [&](size_t bytes) {
      const size_t at = o;
      o = (o + bytes + 127) & ~size_t(127);
      return at;
    };
    p.nslots = ns;
    p.off_x = take(std::max((size_t)H * 4, (size_t)NE * fr.ng_i * kLimbWords * 4));
    p.off_xq4 = take(need4 ? (size_t)fr.ng_h * kLimbWords * 4 : 0);
    p.off_xq2 = take(need2 ? (size_t)fr.ng_h * kLimbWords * 4 : 0);
    p.off_xe4 = take((size_t)fr.ng_h * 8);
    p.off_xe2 = take((size_t)fr.ng_h * 8);
    p.off_ae = take((size_t)NE * fr.ng_i * 8);
    p.off_gu = take((size_t)ns * p.slot_bytes);
    for (int e = 0; e < NE; ++e) {
      const Fmt& f = (has_shared && e == 0) ? fs : fr;
      p.off_dn[e] = take((size_t)p.rows_d * f.d_row);
    }
    p.off_part = take((size_t)2 * p.rows_gu * mh.chunks * 4);
    p.off_pd = take((size_t)NE * p.rows_d * mi.chunks * 4);
    p.off_logits = take((size_t)(E + 1) * 4);
    p.off_bar = take((size_t)(ns + NE) * 8);
    p.total = o;
    if (p.total <= budget) {
      *out = p;
      return true;
    }
  }
  return false;
}

cudaError_t launch_fused(const FusedArgs& a, cudaStream_t s) {
  static int configured_bytes = -1;
  const int bytes = (int)a.plan.total;
  if (bytes > 48 * 1024 && bytes > configured_bytes) {
    cudaError_t e = cudaFuncSetAttribute(fused_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    configured_bytes = bytes;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.plan.P);
  cfg.blockDim = dim3(kBlock);
  cfg.dynamicSmemBytes = (size_t)bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fused_decode_kernel, a);
}

}  // namespace moe
