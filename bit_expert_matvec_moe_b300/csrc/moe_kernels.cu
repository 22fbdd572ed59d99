// Multi-kernel MoE path (any batch) and the kernels behind moe_pack_weights,
// moe_route and moe_expert_forward.  The single-token layer has its own fused
// kernel (moe_decode_b1.cu); both use the device blocks of moe_device.cuh.
#include "moe_internal.h"

namespace moe {

// ---------------------------------------------------------------------------
// moe_pack_weights: canonical (codes, scales, biases) x 3 -> one blob
// ---------------------------------------------------------------------------
// One thread per 4-byte word of the blob.  Gate row i and up row i sit side by
// side (one activation read serves both), each row is its codes (in the order
// described in moe_device.cuh) followed by one (scale | bias << 16) word per
// group, padded to 16 bytes; down rows follow.
__device__ __forceinline__ uint32_t packed_code_word(const uint8_t* crow, int bits, int ng, int o) {
  if (bits == 4) {
    // output byte o: chunk k of up to 32 groups, half h, chunk-local group i
    const int k = o >> 10, rem = o & 1023;
    const int n = min(32, ng - 32 * k);
    const int h = rem / (16 * n), i = (rem % (16 * n)) >> 4, jb = rem & 15;
    const int g = 32 * k + i;
    return *reinterpret_cast<const uint32_t*>(crow + 32 * g + 16 * h + jb);
  }
  // 2-bit: word o/4 of the row holds inputs 16m..16m+15 (m = o/4); field t of
  // byte j takes input 16m + P(j, t), P = {2j, 2j+1, 8+2j, 9+2j}
  const uint32_t cw = *reinterpret_cast<const uint32_t*>(crow + o);  // canonical: input u at bits 2u
  uint32_t out = 0u;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int u[4] = {2 * j, 2 * j + 1, 8 + 2 * j, 9 + 2 * j};
#pragma unroll
    for (int t = 0; t < 4; ++t) out |= ((cw >> (2 * u[t])) & 3u) << (8 * j + 2 * t);
  }
  return out;
}

__global__ void pack_kernel(PackArgs a) {
  const Fmt f = a.f;
  const size_t nwords = f.total / 4;
  for (size_t wi = blockIdx.x * (size_t)blockDim.x + threadIdx.x; wi < nwords; wi += (size_t)gridDim.x * blockDim.x) {
    const size_t off = wi * 4;
    int m, row, inrow, codes_bytes, ng;
    if (off < f.d_off) {
      row = (int)(off / f.gu_pair);
      int rem = (int)(off % f.gu_pair);
      m = rem / f.gu_row;  // 0 gate, 1 up
      inrow = rem % f.gu_row;
      codes_bytes = f.gu_codes;
      ng = f.ng_h;
    } else {
      const size_t o2 = off - f.d_off;
      row = (int)(o2 / f.d_row);
      inrow = (int)(o2 % f.d_row);
      m = 2;
      codes_bytes = f.d_codes;
      ng = f.ng_i;
    }
    uint32_t v = 0u;
    if (inrow < codes_bytes) {
      v = packed_code_word(a.codes[m] + (size_t)row * codes_bytes, f.bits, ng, inrow);
    } else if (inrow < codes_bytes + 4 * ng) {
      const int g = (inrow - codes_bytes) / 4;
      v = (uint32_t)a.scales[m][(size_t)row * ng + g] | ((uint32_t)a.biases[m][(size_t)row * ng + g] << 16);
    }
    *reinterpret_cast<uint32_t*>(a.dst + off) = v;
  }
}

// ---------------------------------------------------------------------------
// RMSNorm (optional) + limbs of each token vector
// ---------------------------------------------------------------------------
// grid = B, block = kBlock.  in fp32 [B, n]; when do_norm, xn = in * rsqrt(mean(in^2)+eps) * gamma
// is written to xn_out; the limbs of (do_norm ? xn : in) go to q (row b at
// q + b * ng * 128 bytes) and the group factors to e.
__global__ void __launch_bounds__(kBlock) norm_quant_kernel(NormQuantArgs a) {
  extern __shared__ float4 nq_smem[];
  float* v = reinterpret_cast<float*>(nq_smem);
  __shared__ float red[kBlock / 32];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const float* src = a.in + (size_t)b * a.n;
  float ss = 0.f;
  for (int i = tid; i < a.n; i += blockDim.x) {
    const float x = src[i];
    v[i] = x;
    ss = fmaf(x, x, ss);
  }
  if (a.do_norm) {
    ss = warp_sum(ss);
    if (lane == 0) red[wid] = ss;
    __syncthreads();
    if (tid == 0) {
      float t = 0.f;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
      red[0] = 1.0f / sqrtf(t / (float)a.n + a.eps);
    }
    __syncthreads();
    const float r = red[0];
    for (int i = tid; i < a.n; i += blockDim.x) {
      float x = v[i] * r;
      if (a.gamma) x *= bf16lo(a.gamma[i]);
      v[i] = x;
      if (a.xn_out) a.xn_out[(size_t)b * a.n + i] = x;
    }
  }
  __syncthreads();
  const int ng = a.n / kGroup;
  bool ok = true;
  uint8_t* qb = a.q + (size_t)b * ng * kLimbBytes;
  for (int g = wid; g < ng; g += blockDim.x >> 5) {
    const float x0 = v[g * kGroup + 2 * lane], x1 = v[g * kGroup + 2 * lane + 1];
    ok &= quantize_group(x0, x1, lane, qb + 16 * g, 16 * ng, a.e + (size_t)b * ng + g);
  }
  if (!ok && lane == 0) atomicOr(&a.hdr->status, ST_NONFINITE);
}

// ---------------------------------------------------------------------------
// router matvec: logits[b][e] = router[e] . xn[b] (+ offset[b][e]); row E is the
// shared-expert gate vector when present (no offset)
// ---------------------------------------------------------------------------
// One warp per router row, tokens in register tiles of 8.  Lane l reads bf16
// elements [8l + 256 s, 8l + 256 s + 8) at step s; partial sums are combined by
// a fixed butterfly, so results do not depend on scheduling.
__global__ void __launch_bounds__(256) router_kernel(RouterArgs a) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int nrows = a.E + (a.gate ? 1 : 0);
  if (row >= nrows) return;
  const uint16_t* R = row < a.E ? a.router + (size_t)row * a.H : a.gate;
  for (int b0 = 0; b0 < a.B; b0 += 8) {
    float acc[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) acc[t] = 0.f;
    for (int c = 8 * lane; c < a.H; c += 256) {
      const uint4 rw = *reinterpret_cast<const uint4*>(R + c);
      const float r[8] = {bf16lo(rw.x), bf16hi(rw.x), bf16lo(rw.y), bf16hi(rw.y),
                          bf16lo(rw.z), bf16hi(rw.z), bf16lo(rw.w), bf16hi(rw.w)};
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        if (b0 + t < a.B) {
          const float4* x4 = reinterpret_cast<const float4*>(a.xn + (size_t)(b0 + t) * a.H + c);
          const float4 xa = x4[0], xb = x4[1];
          float s = acc[t];
          s = fmaf(r[0], xa.x, s); s = fmaf(r[1], xa.y, s); s = fmaf(r[2], xa.z, s); s = fmaf(r[3], xa.w, s);
          s = fmaf(r[4], xb.x, s); s = fmaf(r[5], xb.y, s); s = fmaf(r[6], xb.z, s); s = fmaf(r[7], xb.w, s);
          acc[t] = s;
        }
      }
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const float s = warp_sum(acc[t]);
      const int b = b0 + t;
      if (lane == 0 && b < a.B) {
        float v = s;
        if (row < a.E && a.offset) v += a.offset[(size_t)b * a.E + row];
        a.logits[(size_t)b * (a.E + 1) + row] = v;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// softmax / top-K / renormalise per token: one warp per token
// ---------------------------------------------------------------------------
constexpr int kTopkPer = 32;  // experts per lane: up to 1024 experts
__global__ void __launch_bounds__(32) topk_kernel(TopkArgs a) {
  const int b = blockIdx.x, lane = threadIdx.x;
  const float* lg = a.logits + (size_t)b * (a.E + 1);
  uint32_t key[kTopkPer];
  bool finite = true;
#pragma unroll
  for (int i = 0; i < kTopkPer; ++i) {
    const int e = lane + 32 * i;
    key[i] = 0u;
    if (e < a.E) {
      const float v = lg[e];
      finite &= isfinite(v);
      key[i] = fkey(v);
      if (a.logits_out) a.logits_out[(size_t)b * a.E + e] = v;
    }
  }
  __shared__ int s_idx[kMaxTopK];
  __shared__ float s_val[kMaxTopK], s_w[kMaxTopK];
  warp_topk<kTopkPer>(key, a.K, lane, s_idx, s_val);
  const bool ok = __all_sync(0xffffffffu, finite);
  if (lane == 0) {
    chosen_softmax(s_val, a.K, s_w);
    for (int k = 0; k < a.K; ++k) {
      a.idx[(size_t)b * a.K + k] = s_idx[k];
      a.w[(size_t)b * a.K + k] = s_w[k];
      if (a.idx_out) a.idx_out[(size_t)b * a.K + k] = s_idx[k];
      if (a.w_out) a.w_out[(size_t)b * a.K + k] = s_w[k];
    }
    if (a.gs) a.gs[b] = a.has_gate ? 1.0f / (1.0f + expf(-lg[a.E])) : 1.0f;
    if (!ok) atomicOr(&a.hdr->status, ST_NONFINITE);
  }
}

// ---------------------------------------------------------------------------
// token -> expert grouping (one block): every touched expert is listed once,
// ascending by id, with its (token, slot) entries ascending by token; the shared
// expert, when present, is the last item and holds every token at slot K.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kBlock) bucket_kernel(BucketArgs a) {
  extern __shared__ int bk_smem[];
  int* cnt = bk_smem;            // [E]
  int* off = cnt + a.E;          // [E + 1]
  const int n = a.B * a.K;
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) atomicAdd(&cnt[a.idx[i]], 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0, u = 0;
    for (int e = 0; e < a.E; ++e) {
      off[e] = run;
      if (cnt[e] > 0) {
        a.uniq_e[u] = e;
        a.uniq_off[u] = run;
        ++u;
      }
      run += cnt[e];
    }
    off[a.E] = run;
    int nu = u;
    if (a.has_shared) {
      a.uniq_e[u] = -1;  // shared expert
      a.uniq_off[u] = run;
      nu = u + 1;
      run += a.B;
    }
    a.uniq_off[nu] = run;
    *a.n_uniq = nu;
  }
  __syncthreads();
  // entry i = (b, k): its position among entries of the same expert is the
  // number of earlier entries (in (b, k) order) with that expert
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int e = a.idx[i];
    int pos = 0;
    for (int j = 0; j < i; ++j) pos += (a.idx[j] == e);
    const int b = i / a.K, k = i % a.K;
    a.ent[off[e] + pos] = b * a.nslots + k;
  }
  if (a.has_shared)
    for (int b = threadIdx.x; b < a.B; b += blockDim.x) a.ent[off[a.E] + b] = b * a.nslots + a.K;
}

// ---------------------------------------------------------------------------
// dot products of `nrows` quantised rows with one activation vector
// ---------------------------------------------------------------------------
//   rows      row r starts at rows + row_off(r) (codes, then one (s,b) word per group)
//   xq, xe    the vector's limbs (ng groups, layout of moe_device.cuh) and factors
//   part      out: part[r * chunks + chunk] = partial dot over the chunk's groups
// All warps of the block take part; the caller syncs after.
template <int BITS, typename RowOff>
__device__ __forceinline__ void rows_dot(const uint8_t* rows, RowOff row_off, int nrows, int ng, int codes_bytes,
                                         const uint8_t* xq, const float2* xe, float* part, int wi, int nw, int lane) {
  const RowMap m = make_rowmap(ng);
  const int chunk = wi % m.chunks;
  const int stream = wi / m.chunks;
  const int nstreams = nw / m.chunks;
  if (stream >= nstreams) return;
  const int sub = lane % m.lpr, slot = lane / m.lpr;
  const int g = chunk * 32 + sub;
  const bool gact = g < ng;
  Limbs L;
  float2 es = make_float2(0.f, 0.f);
  if (gact) {
    load_limbs(xq, ng, g, L);
    es = xe[g];
  } else {
    zero_limbs(L);
  }
  const int step = nstreams * m.rpp;
  for (int base = stream * m.rpp; base < nrows; base += step) {
    const int r = base + slot;
    float v = 0.f;
    if (gact && r < nrows) v = row_group<BITS>(rows + row_off(r), ng, codes_bytes, g, L, es);
    v = row_reduce(v, m.lpr);
    if (sub == 0 && r < nrows) part[r * m.chunks + chunk] = v;
  }
}

// ---------------------------------------------------------------------------
// grouped gate/up + SwiGLU: a[b][slot][r] = silu(Wg_r . xn_b) * (Wu_r . xn_b)
// ---------------------------------------------------------------------------
// grid = (row blocks of kRowsGU gate/up row pairs, work items); block = kBlock.
// Item u is expert uniq_e[u] (or the shared expert) with its token entries.
// Without a list (single-expert mode) the item is `blob` with tokens 0..B-1.
template <int BITS>
__device__ void gateup_item(const GateUpArgs& a, const uint8_t* blob, const Fmt& f, const int* ent, int nent) {
  __shared__ float part[2 * kRowsGU * 4];  // up to 4 chunks (hidden <= 8192)
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int r0 = blockIdx.x * kRowsGU;
  const int nr = min(kRowsGU, f.I - r0);
  if (nr <= 0) return;
  const RowMap m = make_rowmap(f.ng_h);
  const uint8_t* rows = blob + (size_t)r0 * f.gu_pair;
  auto off = [&](int r) { return (size_t)(r >> 1) * f.gu_pair + (size_t)(r & 1) * f.gu_row; };
  for (int t = 0; t < nent; ++t) {
    const int e = ent ? ent[t] : t * a.nslots;  // b * nslots + slot
    const int b = e / a.nslots;
    rows_dot<BITS>(rows, off, 2 * nr, f.ng_h, f.gu_codes, a.xq + (size_t)b * f.ng_h * kLimbBytes,
                   a.xe + (size_t)b * f.ng_h, part, wid, nw, lane);
    __syncthreads();
    if ((int)threadIdx.x < nr) {
      const int r = threadIdx.x;
      float g = 0.f, u = 0.f;
      for (int c = 0; c < m.chunks; ++c) {
        g += part[(2 * r) * m.chunks + c];
        u += part[(2 * r + 1) * m.chunks + c];
      }
      a.a_out[(size_t)e * f.I + r0 + r] = silu_mul(g, u);
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kBlock) gateup_kernel(GateUpArgs a) {
  int item = blockIdx.y;
  const uint8_t* blob;
  const int* ent = nullptr;
  int nent;
  int bits;
  if (a.uniq_e == nullptr) {
    if (item > 0) return;
    blob = a.blob;
    nent = a.B;
    bits = a.bits;
  } else {
    if (item >= *a.n_uniq) return;
    const int e = a.uniq_e[item];
    blob = e >= 0 ? a.experts + (size_t)e * a.stride : a.shared;
    bits = e >= 0 ? a.bits : a.shared_bits;
    ent = a.ent + a.uniq_off[item];
    nent = a.uniq_off[item + 1] - a.uniq_off[item];
  }
  const Fmt f = make_fmt(bits, a.H, a.I);
  if (bits == 4)
    gateup_item<4>(a, blob, f, ent, nent);
  else
    gateup_item<2>(a, blob, f, ent, nent);
}

// ---------------------------------------------------------------------------
// grouped down: d[b][slot][j] = Wd_j . a[b][slot]
// ---------------------------------------------------------------------------
template <int BITS>
__device__ void down_item(const DownArgs& a, const uint8_t* blob, const Fmt& f, const int* ent, int nent) {
  __shared__ float part[kRowsD * 4];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int j0 = blockIdx.x * kRowsD;
  const int nr = min(kRowsD, f.H - j0);
  if (nr <= 0) return;
  const RowMap m = make_rowmap(f.ng_i);
  const uint8_t* rows = blob + f.d_off + (size_t)j0 * f.d_row;
  auto off = [&](int r) { return (size_t)r * f.d_row; };
  for (int t = 0; t < nent; ++t) {
    const int e = ent ? ent[t] : t * a.nslots;
    rows_dot<BITS>(rows, off, nr, f.ng_i, f.d_codes, a.aq + (size_t)e * f.ng_i * kLimbBytes, a.ae + (size_t)e * f.ng_i,
                   part, wid, nw, lane);
    __syncthreads();
    for (int r = threadIdx.x; r < nr; r += blockDim.x) {
      float s = 0.f;
      for (int c = 0; c < m.chunks; ++c) s += part[r * m.chunks + c];
      a.d_out[(size_t)e * f.H + j0 + r] = s;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kBlock) down_kernel(DownArgs a) {
  int item = blockIdx.y;
  const uint8_t* blob;
  const int* ent = nullptr;
  int nent, bits;
  if (a.uniq_e == nullptr) {
    if (item > 0) return;
    blob = a.blob;
    nent = a.B;
    bits = a.bits;
  } else {
    if (item >= *a.n_uniq) return;
    const int e = a.uniq_e[item];
    blob = e >= 0 ? a.experts + (size_t)e * a.stride : a.shared;
    bits = e >= 0 ? a.bits : a.shared_bits;
    ent = a.ent + a.uniq_off[item];
    nent = a.uniq_off[item + 1] - a.uniq_off[item];
  }
  const Fmt f = make_fmt(bits, a.H, a.I);
  if (bits == 4)
    down_item<4>(a, blob, f, ent, nent);
  else
    down_item<2>(a, blob, f, ent, nent);
}

// ---------------------------------------------------------------------------
// combine: h[b] += sum_k w[b][k] d[b][k] + gs[b] d[b][K]   (fixed order), or
// the single-expert output out[b] = (acc ? out[b] : 0) + row_w[b] d[b][0]
// ---------------------------------------------------------------------------
__global__ void combine_kernel(CombineArgs a) {
  const size_t n = (size_t)a.B * a.H;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int b = (int)(i / a.H), j = (int)(i % a.H);
    const float* d = a.d + (size_t)b * a.nslots * a.H + j;
    if (a.single) {
      const float wt = a.row_w ? a.row_w[b] : 1.0f;
      const float base = a.accumulate ? a.out[i] : 0.f;
      a.out[i] = fmaf(wt, d[0], base);
    } else {
      float acc = 0.f;
      for (int k = 0; k < a.K; ++k) acc = fmaf(a.w[(size_t)b * a.K + k], d[(size_t)k * a.H], acc);
      if (a.has_shared) acc = fmaf(a.gs[b], d[(size_t)a.K * a.H], acc);
      a.out[i] = a.out[i] + acc;
    }
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
cudaError_t launch_pack(const PackArgs& a, cudaStream_t s) {
  const size_t nwords = a.f.total / 4;
  const int grid = (int)std::min<size_t>((nwords + 255) / 256, 148 * 16);
  pack_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_norm_quant(const NormQuantArgs& a, int B, cudaStream_t s) {
  const size_t sm = (size_t)a.n * sizeof(float);
  if (sm > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(norm_quant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
  }
  norm_quant_kernel<<<B, kBlock, sm, s>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_router(const RouterArgs& a, cudaStream_t s) {
  const int rows = a.E + (a.gate ? 1 : 0);
  router_kernel<<<(rows + 7) / 8, 256, 0, s>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_topk(const TopkArgs& a, int B, cudaStream_t s) {
  topk_kernel<<<B, 32, 0, s>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_bucket(const BucketArgs& a, cudaStream_t s) {
  bucket_kernel<<<1, kBlock, (size_t)(2 * a.E + 1) * sizeof(int), s>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_gateup(const GateUpArgs& a, int items, cudaStream_t s) {
  dim3 grid((a.I + kRowsGU - 1) / kRowsGU, items);
  gateup_kernel<<<grid, kBlock, 0, s>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_down(const DownArgs& a, int items, cudaStream_t s) {
  dim3 grid((a.H + kRowsD - 1) / kRowsD, items);
  down_kernel<<<grid, kBlock, 0, s>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) {
  const size_t n = (size_t)a.B * a.H;
  const int grid = (int)std::min<size_t>((n + 255) / 256, 148 * 8);
  combine_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
