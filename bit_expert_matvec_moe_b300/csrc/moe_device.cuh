// Device-side building blocks of the MoE decode path (sm_103a).
//
// Arithmetic scheme of every dequantised matvec
// ---------------------------------------------
// A row of a quantised matrix is split in groups of 64 inputs, each with a bf16
// scale s and bias b, so that W[c] = q[c] * s + b with an unsigned code q
// ("nibble * scale + bias" on the page "397B MoE sur MacBook : 4,4 t/s Moteur
// Flash-MoE", "Techniques de rupture" item 2).  The pages rewrite the product
// (q*s + b)*x as fma(q, s*x, b*x); summed over a group this is the exact identity
//     sum_c (q_c s + b) x_c = s * sum_c q_c x_c + b * sum_c x_c,
// which is what the kernels evaluate.  The activation x of each group is held
// as a 23-bit block-floating-point integer x_c = X_c * 2^e (|X_c| <= 2^22), split
// into three byte limbs X = L2*65536 + L1*256 + L0 (L0, L1 unsigned, L2 signed).
// The group sum sum_c q_c X_c is then exact in int32, computed four products at
// a time with dp4a, and turned into fp32 once per group:
//     dot_g = 2^e * (65536*A2 + 256*A1 + A0),   row += s*dot_g + b*(2^e*sum X).
// The only rounding of the activation is X = rint(x / 2^e), a relative error of
// at most 2^-23 of the group's largest |x|.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

constexpr int kGroup = 64;
constexpr int kLimbWords = 48;  // limb words per group of 64 activations (both widths)
constexpr int kMaxTopK = 8;
constexpr unsigned long long kTimeoutNs = 1000000000ull;  // bounded device waits: 1 s

enum : uint32_t { ST_TIMEOUT = 1u, ST_NONFINITE = 2u };

// Header at offset 0 of every workspace.
struct WsHeader {
  uint32_t status;     // OR of ST_* bits recorded by kernels
  uint32_t abort;      // set when a CTA gave up on a wait; other CTAs leave too
  uint32_t bar_count;  // grid barrier arrivals
  uint32_t bar_gen;    // grid barrier generation
  uint32_t bar_extra;  // test hook: extra arrivals a grid barrier waits for (0 in normal use)
  uint32_t pad[59];
};
static_assert(sizeof(WsHeader) == 256, "header size");

// ---------------------------------------------------------------------------
// packed expert format
// ---------------------------------------------------------------------------
__host__ __device__ inline size_t pad16(size_t x) { return (x + 15) & ~size_t(15); }

struct Fmt {
  int bits, H, I;
  int ng_h, ng_i;          // groups along hidden / inter
  int gu_codes, d_codes;   // code bytes of a gate/up row and of a down row
  int gu_row, d_row;       // padded row strides (codes + (s,b) words)
  int gu_pair;             // gate row + up row
  size_t d_off, total;     // byte offset of the down rows, blob size
};

__host__ __device__ inline Fmt make_fmt(int bits, int H, int I) {
  Fmt f;
  f.bits = bits; f.H = H; f.I = I;
  f.ng_h = H / kGroup; f.ng_i = I / kGroup;
  f.gu_codes = H * bits / 8; f.d_codes = I * bits / 8;
  f.gu_row = (int)pad16((size_t)f.gu_codes + 4 * f.ng_h);
  f.d_row = (int)pad16((size_t)f.d_codes + 4 * f.ng_i);
  f.gu_pair = 2 * f.gu_row;
  f.d_off = (size_t)I * f.gu_pair;
  f.total = f.d_off + (size_t)H * f.d_row;
  return f;
}

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// ---------------------------------------------------------------------------
// block-floating-point limbs of one group of 64 activations (one warp)
// ---------------------------------------------------------------------------
// Lane l holds x[2l] and x[2l+1].  Writes 48 limb words (as bytes) to q and
// (2^e, 2^e * sum X) to *e_s.  Returns false when a value is not finite.
//
// Limb word order, 4-bit codes: for code word m (inputs 8m..8m+7) the six words
//   [L0 even, L0 odd, L1 even, L1 odd, L2 even, L2 odd]; byte j of an "even"
//   word is input 8m+2j, of an "odd" word input 8m+2j+1 (the low / high nibble
//   of code byte j).
// 2-bit codes: for code word m (inputs 16m..16m+15) and field t = 0..3 the
//   three words [L0, L1, L2]; byte j is input 16m+4j+t.
template <int BITS>
__device__ __forceinline__ bool quantize_group(float x0, float x1, int lane, uint8_t* q, float2* e_s) {
  float m = warp_max(fmaxf(fabsf(x0), fabsf(x1)));
  bool finite = isfinite(m);
  int E = 0;
  if (m > 0.f && finite) frexpf(m, &E);  // m = f * 2^E, f in [0.5, 1)
  E = max(E, -100);
  const float up = __uint_as_float((uint32_t)(127 + 22 - E) << 23);   // 2^(22-E)
  const float dn = __uint_as_float((uint32_t)(127 - 22 + E) << 23);   // 2^(E-22)
  int X[2];
  X[0] = finite ? __float2int_rn(x0 * up) : 0;
  X[1] = finite ? __float2int_rn(x1 * up) : 0;
  int s = warp_sum_i(X[0] + X[1]);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c = 2 * lane + h;  // input index within the group
    const int v = X[h];
    const uint8_t l0 = (uint8_t)(v & 255), l1 = (uint8_t)((v >> 8) & 255), l2 = (uint8_t)((v >> 16) & 255);
    int w0, j;  // word index of limb 0, byte within the word, limb stride in words
    int stride;
    if (BITS == 4) {
      const int mw = c >> 3, p = c & 7;
      w0 = 6 * mw + (p & 1);
      j = p >> 1;
      stride = 2;
    } else {
      const int mw = c >> 4, r = c & 15, t = r & 3;
      w0 = 12 * mw + 3 * t;
      j = r >> 2;
      stride = 1;
    }
    q[4 * w0 + j] = l0;
    q[4 * (w0 + stride) + j] = l1;
    q[4 * (w0 + 2 * stride) + j] = l2;
  }
  if (lane == 0) *e_s = make_float2(dn, (float)s * dn);
  return finite;
}

// Exact integer group sum of codes times limbs, returned as an fp32 value
// (before the 2^e factor).  c holds the group's code bytes (32 B 4-bit,
// 16 B 2-bit), L the 48 limb words.
template <int BITS>
__device__ __forceinline__ float group_dot(const uint4 c0, const uint4 c1, const uint32_t (&L)[kLimbWords]) {
  unsigned a0 = 0u, a1 = 0u;
  int a2 = 0;
  if (BITS == 4) {
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const uint32_t lo = w[m] & 0x0F0F0F0Fu, hi = (w[m] >> 4) & 0x0F0F0F0Fu;
      a0 = __dp4a(lo, L[6 * m + 0], a0);
      a0 = __dp4a(hi, L[6 * m + 1], a0);
      a1 = __dp4a(lo, L[6 * m + 2], a1);
      a1 = __dp4a(hi, L[6 * m + 3], a1);
      a2 = __dp4a((int)lo, (int)L[6 * m + 4], a2);
      a2 = __dp4a((int)hi, (int)L[6 * m + 5], a2);
    }
  } else {
    const uint32_t w[4] = {c0.x, c0.y, c0.z, c0.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint32_t qv = (w[m] >> (2 * t)) & 0x03030303u;
        a0 = __dp4a(qv, L[12 * m + 3 * t + 0], a0);
        a1 = __dp4a(qv, L[12 * m + 3 * t + 1], a1);
        a2 = __dp4a((int)qv, (int)L[12 * m + 3 * t + 2], a2);
      }
    }
  }
  return fmaf((float)a2, 65536.f, fmaf((float)a1, 256.f, (float)a0));
}

__device__ __forceinline__ void load_limbs(const uint32_t* src, uint32_t (&L)[kLimbWords]) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < kLimbWords / 4; ++i) {
    const uint4 v = s4[i];
    L[4 * i + 0] = v.x; L[4 * i + 1] = v.y; L[4 * i + 2] = v.z; L[4 * i + 3] = v.w;
  }
}

// Geometry of the lane -> (row, group) mapping for rows of `ng` groups.
struct RowMap {
  int lpr;     // lanes per row chunk (power of two, <= 32)
  int chunks;  // chunks per row (ng > 32 only)
  int rpp;     // rows per warp pass (32 / lpr)
};
__host__ __device__ inline RowMap make_rowmap(int ng) {
  RowMap m;
  int l = 1;
  while (l < ng && l < 32) l <<= 1;
  m.lpr = l;
  m.chunks = (ng + 31) / 32;
  m.rpp = 32 / l;
  return m;
}

// Dot products of `nrows` quantised rows with one activation vector.
//   rows      row r starts at rows + row_off(r) (codes, then one (s,b) word per group)
//   xq, xe    the vector's limbs (ng x 48 words) and (2^e, 2^e sum X) per group
//   part      out: part[r * chunks + chunk] = partial dot over the chunk's groups
// All warps w0 <= w < w0 + nw of the block take part; the caller syncs after.
template <int BITS, typename RowOff>
__device__ __forceinline__ void rows_dot(const uint8_t* rows, RowOff row_off, int nrows, int ng, int codes_bytes,
                                         const uint32_t* xq, const float2* xe, float* part, int wi, int nw, int lane) {
  const RowMap m = make_rowmap(ng);
  if (nw < m.chunks) return;  // caller guarantees enough warps
  const int chunk = wi % m.chunks;
  const int stream = wi / m.chunks;
  const int nstreams = nw / m.chunks;
  if (stream >= nstreams) return;
  const int sub = lane % m.lpr, slot = lane / m.lpr;
  const int g = chunk * 32 + sub;
  const bool gact = g < ng;
  uint32_t L[kLimbWords];
  float2 es = make_float2(0.f, 0.f);
  if (gact) {
    load_limbs(xq + (size_t)g * kLimbWords, L);
    es = xe[g];
  } else {
#pragma unroll
    for (int i = 0; i < kLimbWords; ++i) L[i] = 0u;
  }
  const int step = nstreams * m.rpp;
  for (int base = stream * m.rpp; base < nrows; base += step) {
    const int r = base + slot;
    float v = 0.f;
    if (gact && r < nrows) {
      const uint8_t* row = rows + row_off(r);
      uint4 c0, c1 = make_uint4(0u, 0u, 0u, 0u);
      if (BITS == 4) {
        c0 = *reinterpret_cast<const uint4*>(row + g * 32);
        c1 = *reinterpret_cast<const uint4*>(row + g * 32 + 16);
      } else {
        c0 = *reinterpret_cast<const uint4*>(row + g * 16);
      }
      const uint32_t sb = *reinterpret_cast<const uint32_t*>(row + codes_bytes + 4 * g);
      const float d = group_dot<BITS>(c0, c1, L);
      v = fmaf(bf16lo(sb) * es.x, d, bf16hi(sb) * es.y);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      if (o < m.lpr) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (sub == 0 && r < nrows) part[r * m.chunks + chunk] = v;
  }
}

// ---------------------------------------------------------------------------
// top-K of one token's logits (one block of kThreadsTopK threads)
// ---------------------------------------------------------------------------
// Order-preserving 64-bit key: larger logit first, then smaller index.
__device__ __forceinline__ unsigned long long topk_key(float v, int idx) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)idx);
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// logits: smem [E]; cand: smem scratch of (nwarps * K) keys; outputs written by
// thread 0 into sel_idx[K], sel_w[K].  Returns (to every thread) false when a
// logit is not finite.  Uses at most 8 values per thread (E <= 8 * blockDim).
__device__ inline bool block_topk(const float* logits, int E, int K, unsigned long long* cand, int* sel_idx,
                                  float* sel_w, int* flag) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
  unsigned long long key[8];
  int bad = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = tid + i * blockDim.x;
    if (e < E) {
      const float v = logits[e];
      if (!isfinite(v)) bad = 1;
      key[i] = topk_key(v, e);
    } else {
      key[i] = 0ull;
    }
  }
  if (tid == 0) *flag = 0;
  __syncthreads();
  if (bad) atomicOr(flag, 1);
  // per-warp top-K
  for (int k = 0; k < K; ++k) {
    unsigned long long best = 0ull;
#pragma unroll
    for (int i = 0; i < 8; ++i) best = key[i] > best ? key[i] : best;
    best = warp_max_u64(best);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (key[i] == best) key[i] = 0ull;
    if (lane == 0) cand[wid * K + k] = best;
  }
  __syncthreads();
  if (wid == 0) {
    unsigned long long ck[8];
    const int nc = nw * K;  // <= 16 * 8 = 128 candidates
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = lane + 32 * i;
      ck[i] = c < nc ? cand[c] : 0ull;
    }
    float lv[kMaxTopK];
    int li[kMaxTopK];
    for (int k = 0; k < K; ++k) {
      unsigned long long best = 0ull;
#pragma unroll
      for (int i = 0; i < 8; ++i) best = ck[i] > best ? ck[i] : best;
      best = warp_max_u64(best);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (ck[i] == best) ck[i] = 0ull;
      const int e = (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
      li[k] = e;
      lv[k] = logits[e];
    }
    if (lane == 0) {
      // softmax over all experts renormalised over the chosen ones equals a
      // softmax over the chosen logits only (the common factor cancels)
      float z[kMaxTopK], sum = 0.f;
      for (int k = 0; k < K; ++k) {
        z[k] = expf(lv[k] - lv[0]);
        sum += z[k];
      }
      for (int k = 0; k < K; ++k) {
        sel_idx[k] = li[k];
        sel_w[k] = z[k] / sum;
      }
    }
  }
  __syncthreads();
  return *flag == 0;
}

// ---------------------------------------------------------------------------
// mbarrier + bulk copy (TMA engine, non-tensor form)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// bytes: multiple of 16, both addresses 16-byte aligned, < 2^20 per barrier phase
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on an mbarrier phase; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kTimeoutNs) return false;
  }
  return true;
}

// ---------------------------------------------------------------------------
// grid barrier over a co-resident (cooperative) grid, bounded
// ---------------------------------------------------------------------------
// Thread 0 of each block.  arrive() returns the generation to wait on.
__device__ __forceinline__ uint32_t grid_arrive(WsHeader* hdr, uint32_t nblocks) {
  nblocks += *(volatile uint32_t*)&hdr->bar_extra;
  const uint32_t g = ld_acquire_u32(&hdr->bar_gen);
  __threadfence();
  const uint32_t prev = atomicAdd(&hdr->bar_count, 1u);
  if (prev == nblocks - 1) {
    atomicExch(&hdr->bar_count, 0u);
    __threadfence();
    st_release_u32(&hdr->bar_gen, g + 1u);
  }
  return g;
}
__device__ __forceinline__ bool grid_wait(WsHeader* hdr, uint32_t g) {
  const unsigned long long t0 = globaltimer();
  while (ld_acquire_u32(&hdr->bar_gen) == g) {
    if (*(volatile uint32_t*)&hdr->abort) return false;
    if (globaltimer() - t0 > kTimeoutNs) {
      atomicOr(&hdr->status, ST_TIMEOUT);
      atomicExch(&hdr->abort, 1u);
      return false;
    }
    __nanosleep(20);
  }
  return true;
}

}  // namespace moe
