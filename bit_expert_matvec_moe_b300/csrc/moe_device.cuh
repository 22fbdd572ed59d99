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
// which is what the kernels evaluate: one scale product and one bias product
// per group instead of per weight.
//
// The activation x of each group is held as a 23-bit block-floating-point
// integer x_c ~ X_c * 2^(e-22) with |X_c| <= 2^22 and 2^(e-1) <= max|x| < 2^e,
// split into three byte limbs X = 65536*L2 + 256*L1 + L0 (L0, L1 unsigned, L2
// signed).  The group sum sum_c q_c X_c is then exact in integers, four
// products per dp4a, and turns into fp32 once per group:
//     dot_g = 2^(e-22) * (65536*A2 + 256*A1 + A0),  row += s*dot_g + b*(2^(e-22)*sum X).
// The only rounding of the activation is X = rint(x * 2^(22-e)): an absolute
// error of at most 2^-23 of 2^e, i.e. <= 2^-22 of the group's largest |x|,
// finer than fp32's own rounding of that largest value.
//
// Limb layout (shared by 4-bit and 2-bit codes)
// ---------------------------------------------
// A group of 64 inputs is 8 "words" q = 0..7 of 8 inputs (8q .. 8q+7).  Its
// limbs are 48 32-bit words, six per word q: (L0 even, L0 odd, L1 even, L1 odd,
// L2 even, L2 odd) at 6q .. 6q+5; byte j of an "even" word holds input 8q+2j,
// of an "odd" word input 8q+2j+1.  In memory the 48 words form 12 packs of 16
// bytes, and a vector of ng groups stores pack k of group g at
// [(k * ng + g) * 16 bytes], so that lane g of a warp reads its group's packs
// with conflict-free 16-byte loads.
//
// Packed code layout (moe_pack_weights; opaque to callers)
// --------------------------------------------------------
// 4-bit: a group's 32 code bytes are two 16-byte halves (inputs 0..31, 32..63),
//   byte j of a half = inputs 2j (low nibble) and 2j+1 (high nibble) of that
//   half, as in the canonical layout.  Groups are taken in chunks of up to 32;
//   inside a chunk of n groups all first halves come first, then all second
//   halves: half h of chunk-local group i sits at chunk_base + 16*(h*n + i).
// 2-bit: a group is 16 code bytes = 4 words m = 0..3 of 16 inputs; inside word
//   m, field t (bits 2t..2t+1) of byte j holds input 16m + P(j, t) with
//   P(j,0) = 2j, P(j,1) = 2j+1, P(j,2) = 8+2j, P(j,3) = 9+2j, so that field t
//   pairs with the same limb words as a 4-bit word (t=0,1: word 2m even/odd;
//   t=2,3: word 2m+1 even/odd).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

constexpr int kGroup = 64;
constexpr int kLimbWords = 48;                    // limb words per group of 64 inputs
constexpr int kLimbPacks = kLimbWords / 4;        // 16-byte packs per group
constexpr int kLimbBytes = kLimbPacks * 16;       // 192 bytes per group
constexpr int kMaxTopK = 8;
constexpr int kMaxBars = 16;                      // split grid barriers per workspace
constexpr unsigned long long kTimeoutNs = 1000000000ull;  // bounded device waits: 1 s

enum : uint32_t { ST_TIMEOUT = 1u, ST_NONFINITE = 2u };

// Header at offset 0 of every workspace (256 bytes).  The first 32 bytes are
// the error state (cleared by moe_get_device_status); the launch counter lives
// on across calls.
struct WsHeader {
  uint32_t status;     // OR of ST_* bits recorded by kernels
  uint32_t abort;      // set when a CTA gave up on a wait; other CTAs leave too
  uint32_t rsv[2];
  uint32_t bar_extra;  // test hook: added to the epoch every cross-block wait expects (0 in normal use)
  uint32_t rsv2[3];
  // layers started by the blocks of the single-token kernels: every block adds
  // one per layer (a launch of L layers adds L per block), so the first layer
  // of a launch finds its epoch as count / grid + 1 and layer l of the launch
  // has that epoch + l
  unsigned long long launches;
  // blocks that finished publishing their logits / activations (each layer
  // adds its grid size to each): a hint that lets one thread per block wait on
  // a single word before the epoch-checked reads
  unsigned long long published_logits;
  unsigned long long published_act;
  // blocks of stack launches that published a layer's output rows for the
  // next layer (each such layer adds its grid size); a stack launch reads it
  // at its start and waits for its own layers' increments above that value
  unsigned long long published_h;
};
static_assert(sizeof(WsHeader) == 64, "header size");
constexpr size_t kHeaderErrorBytes = 32;
constexpr size_t kHeaderBytes = 256;

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

// Byte offsets, inside a row's code bytes, of the two 16-byte halves of group g
// (4-bit) or of its single 16-byte block (2-bit, second value unused).
__host__ __device__ inline void group_code_offsets(int bits, int ng, int g, int* o0, int* o1) {
  if (bits == 4) {
    const int k = g >> 5, i = g & 31;
    const int n = min(32, ng - 32 * k);
    *o0 = 1024 * k + 16 * i;
    *o1 = 1024 * k + 16 * (n + i);
  } else {
    *o0 = 16 * g;
    *o1 = 16 * g;
  }
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
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
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

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// dp4a with unsigned a (codes) and unsigned / signed b (limbs)
__device__ __forceinline__ uint32_t dp4a_uu(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// ---------------------------------------------------------------------------
// limbs of one group of 64 activations (one warp)
// ---------------------------------------------------------------------------
// Lane l holds inputs 2l and 2l+1 of the group.  Writes the group's 12 limb
// packs to `packs` (pack k at packs + k * pack_stride bytes) and
// (2^(e-22), 2^(e-22) * sum X) to *es.  Returns false when a value is not finite.
__device__ __forceinline__ bool quantize_group(float x0, float x1, int lane, uint8_t* packs, int pack_stride,
                                               float2* es) {
  const float m = warp_max(fmaxf(fabsf(x0), fabsf(x1)));
  const bool finite = isfinite(m);
  int E = 0;
  if (m > 0.f && finite) frexpf(m, &E);  // m = f * 2^E, f in [0.5, 1)
  E = max(E, -100);
  const float up = __uint_as_float((uint32_t)(127 + 22 - E) << 23);  // 2^(22-E)
  const float dn = __uint_as_float((uint32_t)(127 - 22 + E) << 23);  // 2^(E-22)
  const int X0 = finite ? __float2int_rn(x0 * up) : 0;
  const int X1 = finite ? __float2int_rn(x1 * up) : 0;
  int s = X0 + X1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  // inputs 2l (even) and 2l+1 (odd): word q = l >> 2, byte j = l & 3
  const int q = lane >> 2, j = lane & 3;
  const uint8_t v[6] = {(uint8_t)(X0 & 255),         (uint8_t)(X1 & 255),
                        (uint8_t)((X0 >> 8) & 255),  (uint8_t)((X1 >> 8) & 255),
                        (uint8_t)((X0 >> 16) & 255), (uint8_t)((X1 >> 16) & 255)};
#pragma unroll
  for (int t = 0; t < 6; ++t) {
    const int w = 6 * q + t;
    packs[(w >> 2) * pack_stride + (w & 3) * 4 + j] = v[t];
  }
  if (lane == 0) *es = make_float2(dn, (float)s * dn);
  return finite;
}

// Lane's limbs of group g of a vector with ng groups (smem): 48 registers.
struct Limbs {
  uint32_t w[kLimbWords];
};
__device__ __forceinline__ void load_limbs(const uint8_t* vec, int ng, int g, Limbs& L) {
#pragma unroll
  for (int k = 0; k < kLimbPacks; ++k) {
    const uint4 v = *reinterpret_cast<const uint4*>(vec + ((size_t)k * ng + g) * 16);
    L.w[4 * k + 0] = v.x; L.w[4 * k + 1] = v.y; L.w[4 * k + 2] = v.z; L.w[4 * k + 3] = v.w;
  }
}
__device__ __forceinline__ void zero_limbs(Limbs& L) {
#pragma unroll
  for (int i = 0; i < kLimbWords; ++i) L.w[i] = 0u;
}

// Exact integer group sum sum_c q_c X_c of one group (codes c0, c1 as laid
// out above; c1 unused for 2-bit), returned as an fp32 value before 2^(e-22).
template <int BITS>
__device__ __forceinline__ float group_dot(const uint4 c0, const uint4 c1, const Limbs& L) {
  if (BITS == 4) {
    // low nibbles as bytes, high nibbles in place (bytes 16 * code): the b*
    // sums are exactly 16 times the high-nibble sums, so no shift per word
    uint32_t a0 = 0u, a1 = 0u, b0 = 0u, b1 = 0u;
    int a2 = 0, b2 = 0;
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint32_t lo = w[q] & 0x0F0F0F0Fu, hi = w[q] & 0xF0F0F0F0u;
      a0 = dp4a_uu(lo, L.w[6 * q + 0], a0);
      b0 = dp4a_uu(hi, L.w[6 * q + 1], b0);
      a1 = dp4a_uu(lo, L.w[6 * q + 2], a1);
      b1 = dp4a_uu(hi, L.w[6 * q + 3], b1);
      a2 = dp4a_us(lo, L.w[6 * q + 4], a2);
      b2 = dp4a_us(hi, L.w[6 * q + 5], b2);
    }
    // limbs 0 and 1 combine exactly in int32 (< 2^26); the b parts are
    // multiples of 16, so the shifts are exact
    const int t01 = (int)(a0 + (a1 << 8)) + (int)((b0 + (b1 << 8)) >> 4);
    const int t2 = a2 + (b2 >> 4);
    return fmaf((float)t2, 65536.f, (float)t01);
  } else {
    uint32_t a0 = 0u, a1 = 0u;
    int a2 = 0;
    const uint32_t w[4] = {c0.x, c0.y, c0.z, c0.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      // fields 0, 1 pair with word 2m (even, odd); fields 2, 3 with word 2m+1
      const uint32_t f[4] = {w[m] & 0x03030303u, (w[m] >> 2) & 0x03030303u, (w[m] >> 4) & 0x03030303u,
                             (w[m] >> 6) & 0x03030303u};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int base = 6 * (2 * m + (t >> 1)) + (t & 1);
        a0 = dp4a_uu(f[t], L.w[base + 0], a0);
        a1 = dp4a_uu(f[t], L.w[base + 2], a1);
        a2 = dp4a_us(f[t], L.w[base + 4], a2);
      }
    }
    return fmaf((float)a2, 65536.f, (float)(int)(a0 + (a1 << 8)));
  }
}

// Partial row dot of one lane: group g of a quantised row (codes at `row`,
// one (scale | bias << 16) word per group after `codes_bytes`).
template <int BITS>
__device__ __forceinline__ float row_group(const uint8_t* row, int ng, int codes_bytes, int g, const Limbs& L,
                                           float2 es) {
  int o0, o1;
  group_code_offsets(BITS, ng, g, &o0, &o1);
  const uint4 c0 = *reinterpret_cast<const uint4*>(row + o0);
  uint4 c1 = c0;
  if (BITS == 4) c1 = *reinterpret_cast<const uint4*>(row + o1);
  const uint32_t sb = *reinterpret_cast<const uint32_t*>(row + codes_bytes + 4 * g);
  const float d = group_dot<BITS>(c0, c1, L);
  return fmaf(bf16lo(sb) * es.x, d, bf16hi(sb) * es.y);
}

// Geometry of the lane -> (row, group) mapping for rows of `ng` groups.
struct RowMap {
  int lpr;     // lanes per row chunk (power of two, <= 32)
  int chunks;  // chunks of 32 groups per row
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
// reduce over the lpr lanes of a row (lpr a power of two)
__device__ __forceinline__ float row_reduce(float v, int lpr) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    if (o < lpr) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// top-K of one token's logits by one warp
// ---------------------------------------------------------------------------
// Order-preserving 32-bit key of a float (larger float -> larger key).
__device__ __forceinline__ uint32_t fkey(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Warp-wide top-K over E <= 32*kPer logits held as lane l, slot i <-> expert
// l + 32 i (absent experts hold key 0).  Order: larger logit first, then lower
// index.  Pick k goes to idx[k] and its logit to val[k] (written by lane 0;
// shared or global memory).  The loop over k stays rolled: one warp runs it,
// and a compact body keeps it in the instruction cache.
template <int kPer>
__device__ __forceinline__ void warp_topk(uint32_t (&key)[kPer], int K, int lane, int* idx, float* val) {
  for (int k = 0; k < K; ++k) {
    uint32_t best = 0u;
#pragma unroll
    for (int i = 0; i < kPer; ++i) best = max(best, key[i]);
    const uint32_t top = __reduce_max_sync(0xffffffffu, best);
    int mine = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (key[i] == top) mine = min(mine, lane + 32 * i);
    const int e = (int)__reduce_min_sync(0xffffffffu, (uint32_t)mine);
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (lane + 32 * i == e) key[i] = 0u;
    if (lane == 0) {
      idx[k] = e;
      val[k] = __uint_as_float((top & 0x80000000u) ? (top & 0x7FFFFFFFu) : ~top);
    }
  }
}

// w_k = softmax over all experts renormalised over the chosen ones, computed as
// a softmax over the chosen logits only (the common factor cancels).  One thread.
__device__ __forceinline__ void chosen_softmax(const float* val, int K, float* w) {
  float sum = 0.f;
  for (int k = 0; k < K; ++k) {
    w[k] = expf(val[k] - val[0]);
    sum += w[k];
  }
  for (int k = 0; k < K; ++k) w[k] = w[k] / sum;
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
// Non-blocking test of a phase: cheap when it has already completed (about 50
// cycles on B300 against about 170 for a try_wait that finds it complete).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_test_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kTimeoutNs) return false;
  }
  return true;
}

// ---------------------------------------------------------------------------
// cross-block publication with the flag in the data
// ---------------------------------------------------------------------------
// A published float is one aligned 64-bit word (epoch << 32 | value bits),
// written and read with single 64-bit accesses, which are single-copy atomic:
// a reader that sees the current launch's epoch sees that launch's value, so no
// fence or counter is needed between writer and reader.
__device__ __forceinline__ void st_pub(unsigned long long* p, float v, uint32_t epoch) {
  const unsigned long long w = ((unsigned long long)epoch << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ unsigned long long ld_pub(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ bool pub_ready(unsigned long long w, uint32_t epoch) { return (uint32_t)(w >> 32) == epoch; }
__device__ __forceinline__ float pub_value(unsigned long long w) { return __uint_as_float((uint32_t)w); }

__device__ __forceinline__ void red_relaxed_add_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// One thread: bounded wait (with back-off) until the counter reaches target;
// false on timeout or when another block gave up.
__device__ __forceinline__ bool wait_count(WsHeader* hdr, const unsigned long long* cnt, unsigned long long target) {
  if ((long long)(ld_pub(cnt) - target) >= 0) return true;
  const unsigned long long t0 = globaltimer();
  while ((long long)(ld_pub(cnt) - target) < 0) {
    if (*(volatile uint32_t*)&hdr->abort) return false;
    if (globaltimer() - t0 > kTimeoutNs) {
      atomicOr(&hdr->status, ST_TIMEOUT);
      atomicExch(&hdr->abort, 1u);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

// Bounded poll for n published words p[0], p[stride], ... (n <= 8) of this
// epoch; the values go to out[].  On timeout, or when another block gave up,
// records the error and returns false.
template <int kN>
__device__ __forceinline__ bool poll_pub(WsHeader* hdr, const unsigned long long* p, int stride, int n,
                                         uint32_t epoch, float (&out)[kN]) {
  unsigned long long w[kN];
  bool ready = true;
#pragma unroll
  for (int i = 0; i < kN; ++i) {
    w[i] = i < n ? ld_pub(p + (size_t)i * stride) : ((unsigned long long)epoch << 32);
    ready &= pub_ready(w[i], epoch);
  }
  if (!ready) {
    const unsigned long long t0 = globaltimer();
    int spins = 0;
    while (!ready) {
      ready = true;
#pragma unroll
      for (int i = 0; i < kN; ++i) {
        if (!pub_ready(w[i], epoch)) w[i] = ld_pub(p + (size_t)i * stride);
        ready &= pub_ready(w[i], epoch);
      }
      if (ready) break;
      if ((++spins & 63) == 0) {
        if (*(volatile uint32_t*)&hdr->abort) return false;
        if (globaltimer() - t0 > kTimeoutNs) {
          atomicOr(&hdr->status, ST_TIMEOUT);
          atomicExch(&hdr->abort, 1u);
          return false;
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kN; ++i) out[i] = pub_value(w[i]);
  return true;
}

// named block barrier 1: producers arrive without waiting, the consumer waits
__device__ __forceinline__ void named_arrive(int id, int nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// programmatic dependent launch: let the next kernel on the stream start early,
// and wait for the previous kernel's memory before touching caller data
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_prior() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace moe
