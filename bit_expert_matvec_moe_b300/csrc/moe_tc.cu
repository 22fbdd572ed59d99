// Batched expert contraction on the tcgen05 tensor cores (B > 1).
//
// Work list.  After routing and bucketing (each touched expert once, its
// (token, slot) entries contiguous), tc_plan_kernel cuts every expert's entry
// list into chunks of at most kTcTok entries; a unit of work is one chunk and
// one 128-row tile of that expert's weight rows (gate/up rows interleaved as
// in the packed format, or down rows).
//
// Operands.  tc_pack_kernel writes, for every entry, the B operand rows of
// its activation (fp16 hi and lo rows, inputs permuted inside 8-input chunks,
// one power-of-two scale per entry) - for gate/up from the token's normalised
// hidden state, for down from the entry's SwiGLU activation.
//
// Contraction (tc_contract_kernel, persistent, one 480-thread CTA per SM):
//   warp 0     TMA producer: per unit, the code pieces and (scale, bias) words
//              of 8 groups x 128 rows per stage (3 stages in flight);
//   warp 1     TMA producer: per K-block (64 inputs) the entry rows of B into
//              shared memory (8 K-blocks in flight);
//   warp 2     owns the tensor memory (a ring of 4 accumulators of 64 columns,
//              then one 32-column A block per K slot) and issues, from one
//              elected lane of a warp that walks the work list in step, 4 MMAs
//              (M 128, N 2 x tokens, K 16, A in tensor memory) per K-block,
//              two K-blocks per round of waits, starting a fresh accumulator
//              every kSpanKB K-blocks;
//   warps 3-6  epilogue: add up a unit's partial sums in fp32 registers
//              (one warp per tensor-memory lane quarter), then add hi and lo
//              columns, scale, SwiGLU for gate/up, store;
//   warps 7-14 dequantise the staged codes (fp16 q*s + b) straight into the
//              tensor-memory A blocks: two warps per lane quarter, one taking
//              the even and one the odd K-blocks, each all 64 inputs of its
//              32 rows.
// Waits first test the barrier phase (mbarrier.test_wait, cheap when it has
// already completed) and only then poll with try_wait.  Measured on B300 with
// the 128-token batch: a completed-phase try_wait cost about 170 cycles inside
// the MMA loop, a test_wait about 50; per-MMA descriptor work in a one-lane
// branch cost about 60 cycles an MMA against 45 from a warp-uniform loop.
// Every wait is bounded (1 s); a CTA that gives up records ST_TIMEOUT, lets
// its copies and MMAs in flight finish (bounded), frees its tensor memory and
// returns.  Units are taken round-robin (unit = CTA, CTA + grid, ...), so the
// CTAs working at one time cover all tiles of a few chunks and each expert's
// rows are streamed from HBM once per chunk while B stays in L2.
#include <cuda.h>
#include <cuda_fp16.h>

#include "moe_device.cuh"
#include "moe_internal.h"
#include "moe_tc.cuh"

namespace moe {
namespace tc {

// ---------------------------------------------------------------------------
// work list: chunks of at most kTcTok entries per touched expert
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(32) tc_plan_kernel(TcPlanArgs a) {
  pdl_wait_prior();  // no-op unless launched with programmatic serialisation
  pdl_launch_dependents();
  const int lane = threadIdx.x;
  const int nu = *a.n_uniq;
  int total = 0;
  for (int base = 0; base < nu; base += 32) {
    const int u = base + lane;
    int n = 0, e = 0, e0 = 0;
    if (u < nu) {
      e0 = a.uniq_off[u];
      n = a.uniq_off[u + 1] - e0;
      e = a.uniq_e[u];
    }
    const int nch = (n + kTcTok - 1) / kTcTok;
    int incl = nch;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int first = total + incl - nch;
    for (int c = 0; c < nch; ++c) {
      if (first + c >= a.max_chunks) {
        atomicOr(&a.hdr->status, ST_PLAN);  // cannot happen with a workspace sized for the batch
        break;
      }
      TcChunk ch;
      ch.expert = e;
      ch.e0 = e0 + kTcTok * c;
      ch.n = min(kTcTok, n - kTcTok * c);
      ch.bits = e >= 0 ? a.bits : a.shared_bits;
      a.chunks[first + c] = ch;
    }
    total += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) *a.n_chunks = min(total, a.max_chunks);
}

// Work list of one expert applied to tokens 0 .. B-1 (moe_expert_forward): a
// single item, taken through the shared-expert tensor maps.
__global__ void tc_single_item_kernel(int B, int* n_uniq, int* uniq_e, int* uniq_off, int* ent) {
  pdl_wait_prior();
  pdl_launch_dependents();
  for (int j = threadIdx.x; j < B; j += blockDim.x) ent[j] = j;
  if (threadIdx.x == 0) {
    *n_uniq = 1;
    uniq_e[0] = -1;
    uniq_off[0] = 0;
    uniq_off[1] = B;
  }
}

// ---------------------------------------------------------------------------
// B operand rows: fp16 hi / lo of each entry's activation, scaled per entry
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) tc_pack_kernel(TcPackArgs a) {
  pdl_wait_prior();
  pdl_launch_dependents();
  const int j = blockIdx.x;
  const int total = a.uniq_off[*a.n_uniq];
  if (j >= total) return;
  const int id = a.ent[j];
  if (id < 0 || id >= a.n_ids) {  // cannot happen with a consistent work list
    if (threadIdx.x == 0) atomicOr(&a.hdr->status, ST_BOUNDS);
    return;
  }
  const float* src = a.src + (size_t)(a.by_token ? id / a.nslots : id) * a.K;
  __shared__ float red[8];
  float m = 0.f;
  int bad = 0;
  for (int i = threadIdx.x * 4; i < a.K; i += 256 * 4) {
    const float4 v = *reinterpret_cast<const float4*>(src + i);
    bad |= !isfinite(v.x) | !isfinite(v.y) | !isfinite(v.z) | !isfinite(v.w);
    m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  bad = __syncthreads_or(bad);
  m = red[0];
  for (int w = 1; w < 8; ++w) m = fmaxf(m, red[w]);
  int e = 0;
  if (bad) {
    if (threadIdx.x == 0) atomicOr(&a.hdr->status, ST_NONFINITE);
  } else if (m > 0.f) {
    e = ilogbf(m) - 14;  // max |x| * 2^-e in [2^14, 2^15)
  }
  if (threadIdx.x == 0) a.scale[j] = ldexpf(1.f, e);
  __half* hi = a.dst + (size_t)(2 * j) * a.K;
  __half* lo = hi + a.K;
  for (int c = threadIdx.x; c < a.K / 8; c += 256) {
    const float4 v0 = *reinterpret_cast<const float4*>(src + 8 * c);
    const float4 v1 = *reinterpret_cast<const float4*>(src + 8 * c + 4);
    const float x[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    __align__(16) __half h[8], l[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const float s = ldexpf(x[chunk_perm(p)], -e);
      h[p] = __float2half_rn(s);
      l[p] = __float2half_rn(s - __half2float(h[p]));
    }
    *reinterpret_cast<uint4*>(hi + 8 * c) = *reinterpret_cast<const uint4*>(h);
    *reinterpret_cast<uint4*>(lo + 8 * c) = *reinterpret_cast<const uint4*>(l);
  }
}

// ---------------------------------------------------------------------------
// dequantisation of code words into fp16 pairs (see the header for the order)
// ---------------------------------------------------------------------------
__device__ __forceinline__ __half2 h2bits(uint32_t u) {
  __half2 h;
  memcpy(&h, &u, 4);
  return h;
}
__device__ __forceinline__ uint32_t bits_h2(__half2 h) {
  uint32_t u;
  memcpy(&u, &h, 4);
  return u;
}
// One field spec (moe_tc.cuh) applied to a code word: an fp16 pair q*s + b,
// each rounded once.
__device__ __forceinline__ uint32_t field_to_w(uint32_t w, const FieldSpec f, __half2 s, __half2 b) {
  const __half2 t = h2bits(((w >> f.shift) & f.mask) | kMagic1024);
  const __half2 q = __hfma2(t, h2bits(f.inv_m), h2bits(f.neg_off));
  return bits_h2(__hfma2(q, s, b));
}
// 4-bit word (inputs 8m .. 8m+7 of a group) -> one 8-input chunk
__device__ __forceinline__ uint4 dequant_word4(uint32_t w, __half2 s, __half2 b) {
  return make_uint4(field_to_w(w, kField4[0], s, b), field_to_w(w, kField4[1], s, b), field_to_w(w, kField4[2], s, b),
                    field_to_w(w, kField4[3], s, b));
}
// 2-bit word (inputs 16m .. 16m+15) -> two 8-input chunks
__device__ __forceinline__ void dequant_word2(uint32_t w, __half2 s, __half2 b, uint4& c0, uint4& c1) {
  c0 = make_uint4(field_to_w(w, kField2[0], s, b), field_to_w(w, kField2[1], s, b), field_to_w(w, kField2[2], s, b),
                  field_to_w(w, kField2[3], s, b));
  c1 = make_uint4(field_to_w(w, kField2[4], s, b), field_to_w(w, kField2[5], s, b), field_to_w(w, kField2[6], s, b),
                  field_to_w(w, kField2[7], s, b));
}

// ---------------------------------------------------------------------------
// the contraction
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile("{ .reg .pred p; elect.sync _|p, 0xffffffff; selp.u32 %0, 1, 0, p; }" : "=r"(pred));
  return pred != 0;
}
// Bounded mbarrier wait that also gives up once another role of the CTA has.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort) {
  if (mbar_test_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (globaltimer() - t0 > kTimeoutNs) {
      *abort = 1u;
      return false;
    }
  }
  return true;
}
// The same for a whole warp: true only if every lane saw the phase complete.
__device__ __forceinline__ bool tc_wait_warp(uint64_t* bar, uint32_t parity, volatile uint32_t* abort) {
  return __all_sync(0xffffffffu, tc_wait(bar, parity, abort));
}
// After a give-up: wait (bounded, whatever the abort flag says) for the last
// `issued` phases of a ring of `slots` barriers armed by this thread, so that
// no copy is still writing into shared memory when the CTA leaves.
__device__ __forceinline__ void drain_ring(uint64_t* ring, int slots, uint32_t issued) {
  const uint32_t n = issued < (uint32_t)slots ? issued : (uint32_t)slots;
  for (uint32_t k = issued - n; k < issued; ++k) mbar_wait(&ring[k % slots], (k / slots) & 1u);
}

__global__ void __launch_bounds__(kTcThreads, 1)
    tc_contract_kernel(const __grid_constant__ CUtensorMap m_codes, const __grid_constant__ CUtensorMap m_sb,
                       const __grid_constant__ CUtensorMap m_codes_sh, const __grid_constant__ CUtensorMap m_sb_sh,
                       const __grid_constant__ CUtensorMap m_b, const TcContractArgs a) {
  extern __shared__ __align__(1024) uint8_t tc_raw[];
  uint8_t* sm = tc_raw + ((1024u - (su32(tc_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBars);
  uint64_t* full_c = bars;                   // code stage landed (TMA bytes)
  uint64_t* empty_c = full_c + kCodeSlots;   // code stage read by the 8 dequantising warps
  // K slot ready: the 4 dequantising warps of its parity have written A and
  // the B copy has landed (the B producer's expect_tx is the fifth arrival)
  uint64_t* full_a = empty_c + kCodeSlots;
  uint64_t* empty_k = full_a + kKSlots;      // K-block read by the MMAs (commit)
  uint64_t* dfull = empty_k + kKSlots;       // partial sum complete (commit)
  uint64_t* dempty = dfull + kDBufs;         // partial sum read by the 4 epilogue warps
  uint64_t* drain = dempty + kDBufs;
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + kOffMisc);  // [0] tensor memory, [1] abort, [2] status bits
  volatile uint32_t* abort = misc + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kCodeSlots; ++i) {
      mbar_init(&full_c[i], 1);
      mbar_init(&empty_c[i], 8);
    }
    for (int i = 0; i < kKSlots; ++i) {
      mbar_init(&full_a[i], 5);
      mbar_init(&empty_k[i], 1);
    }
    for (int i = 0; i < kDBufs; ++i) {
      mbar_init(&dfull[i], 1);
      mbar_init(&dempty[i], 4);
    }
    mbar_init(drain, 1);
    misc[1] = 0u;
    misc[2] = 0u;
    fence_mbar_init();
  }
  if (warp == kWarpCodes && lane == 0) {
    prefetch_tmap(&m_codes);
    prefetch_tmap(&m_sb);
    prefetch_tmap(&m_codes_sh);
    prefetch_tmap(&m_sb_sh);
    prefetch_tmap(&m_b);
  }
  constexpr uint32_t kCols = kTmemCols;
  if (warp == kWarpMma) {
    tmem_alloc(&misc[0], kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  // set-up above overlaps the previous kernel when launched with programmatic
  // serialisation; nothing it wrote is read before this wait
  pdl_wait_prior();
  pdl_launch_dependents();
  const int n_units = *a.n_chunks * a.tiles;
  const int nst = (a.ng + kStageGroups - 1) / kStageGroups;

  if (warp == kWarpCodes) {
    // ---- code / (scale, bias) stages ------------------------------------
    if (lane == 0) {
      uint32_t cc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const TcChunk ch = a.chunks[u / a.tiles];
        const int row0 = (u % a.tiles) * kTcM;
        const bool sh = ch.expert < 0;
        const CUtensorMap* mc = sh ? &m_codes_sh : &m_codes;
        const CUtensorMap* ms = sh ? &m_sb_sh : &m_sb;
        const int z = sh ? 0 : ch.expert;
        const int code_bytes = a.ng * 8 * ch.bits;  // 64 inputs x bits / 8 per group
        const uint32_t tx = (ch.bits == 4 ? 2u : 1u) * kHalfBoxBytes + kSbBoxBytes;
        for (int st = 0; st < nst; ++st, ++cc) {
          const uint32_t slot = cc % kCodeSlots;
          if (!(ok = tc_wait(&empty_c[slot], ((cc / kCodeSlots) & 1u) ^ 1u, abort))) break;
          uint8_t* dst = sm + kOffCodes + slot * kCodeSlotBytes;
          int x0, x1;
          stage_code_x(ch.bits, a.ng, st, &x0, &x1);
          mbar_expect_tx(&full_c[slot], tx);
          tma_load_3d(dst, mc, x0, row0, z, &full_c[slot]);
          if (ch.bits == 4) tma_load_3d(dst + kHalfBoxBytes, mc, x1, row0, z, &full_c[slot]);
          tma_load_3d(dst + 2 * kHalfBoxBytes, ms, code_bytes + 32 * st, row0, z, &full_c[slot]);
        }
      }
      drain_ring(full_c, kCodeSlots, cc);
    }
    __syncwarp();
  } else if (warp == kWarpB) {
    // ---- activation K-blocks ---------------------------------------------
    if (lane == 0) {
      uint32_t kc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const TcChunk ch = a.chunks[u / a.tiles];
        const int boxes = (ch.n + 7) >> 3;
        for (int kb = 0; kb < a.ng; ++kb, ++kc) {
          const uint32_t slot = kc % kKSlots;
          if (!(ok = tc_wait(&empty_k[slot], ((kc / kKSlots) & 1u) ^ 1u, abort))) break;
          uint8_t* dst = sm + kOffK + slot * kKSlotBytes;
          mbar_expect_tx(&full_a[slot], (uint32_t)boxes * kBBoxBytes);
          for (int i = 0; i < boxes; ++i)
            tma_load_2d(dst + i * kBBoxBytes, &m_b, kb * 64, 2 * ch.e0 + (int)kBBoxRows * i, &full_a[slot]);
        }
      }
      // (the slots' phases also wait for the dequantising warps; after a give-up
      // the bounded wait then just outlasts the copies in flight)
      drain_ring(full_a, kKSlots, kc);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ---- MMAs ---------------------------------------------------------------
    // The whole warp walks the work list (so every operand below is
    // warp-uniform); one elected lane issues the MMAs and commits.  Partial
    // sums: a fresh accumulator (ring slot pc % kDBufs) every kSpanKB K-blocks
    // of a unit, committed to dfull for the epilogue.
    uint32_t kc = 0, pc = 0;
    bool ok = true;
    const uint64_t bdesc0 = sdesc_sw128_kmajor(su32(sm + kOffK));
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const TcChunk ch = a.chunks[u / a.tiles];
      const uint32_t idesc = make_idesc_f16(kTcM, 2 * ((ch.n + 7) & ~7));
      for (int kb0 = 0; kb0 < a.ng && ok; kb0 += kSpanKB, ++pc) {
        const uint32_t d = pc % kDBufs;
        if (!(ok = __all_sync(0xffffffffu, lane != 0 || tc_wait(&dempty[d], ((pc / kDBufs) & 1u) ^ 1u, abort)))) break;
        tc_fence_after();
        const uint32_t dt = tmem + d * kDCols;
        const int kb1 = min(a.ng, kb0 + kSpanKB);
        // K-blocks in pairs: one round of waits, then up to 8 MMAs
        for (int kb = kb0, nkb = 0; kb < kb1; kb += nkb, kc += nkb) {
          nkb = min(2, kb1 - kb);
          bool w = true;
          if (lane == 0) {
            for (int i = 0; i < nkb && w; ++i) {
              const uint32_t sl = (kc + i) % kKSlots, pa = ((kc + i) / kKSlots) & 1u;
              w = tc_wait(&full_a[sl], pa, abort);
            }
          }
          if (!(ok = __all_sync(0xffffffffu, w))) break;
          tc_fence_after();
          if (elect_one()) {
            for (int i = 0; i < nkb; ++i) {
              const uint32_t slot = (kc + i) % kKSlots;
              const uint64_t bd = bdesc0 + (uint64_t)(slot * (kKSlotBytes >> 4));
              const uint32_t at = tmem + kTmemACol0 + slot * 32;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_f16_ts(dt, at + 8 * kk, bd + 2 * kk, idesc, (kb + i != kb0 || kk != 0) ? 1u : 0u);
              mma_commit(&empty_k[slot]);
            }
          }
          __syncwarp();
        }
        if (ok && elect_one()) mma_commit(&dfull[d]);
        __syncwarp();
      }
    }
    // every MMA issued by this CTA has finished reading its operands
    if (elect_one()) {
      mma_commit(drain);
      mbar_wait(drain, 0);
    }
    __syncwarp();
  } else if (warp < kWarpDeq0) {
    // ---- epilogue: partial sums -> outputs ------------------------------------
    const int q = warp & 3;
    uint32_t pc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const TcChunk ch = a.chunks[u / a.tiles];
      const int row = (u % a.tiles) * kTcM + 32 * q + lane;
      const int n8 = (ch.n + 7) & ~7;
      // this lane's row: token t's hi + lo sum, added up over the unit's partials
      float acc[kTcTok];
#pragma unroll
      for (int t = 0; t < kTcTok; ++t) acc[t] = 0.f;
      for (int kb0 = 0; kb0 < a.ng; kb0 += kSpanKB, ++pc) {
        const uint32_t d = pc % kDBufs;
        if (!(ok = tc_wait_warp(&dfull[d], (pc / kDBufs) & 1u, abort))) break;
        tc_fence_after();
        const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + d * kDCols;
        uint32_t v[4][16];
#pragma unroll
        for (int cb = 0; cb < 4; ++cb)
          if (8 * cb < n8) tmem_ld16(ta + 16 * cb, v[cb]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&dempty[d]);
#pragma unroll
        for (int cb = 0; cb < 4; ++cb)
          if (8 * cb < n8) {
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[8 * cb + i] += __uint_as_float(v[cb][2 * i]) + __uint_as_float(v[cb][2 * i + 1]);
          }
      }
      if (!ok) break;
#pragma unroll
      for (int t = 0; t < kTcTok; ++t) {
        if (t < ch.n) {
          const int j = ch.e0 + t;
          const int id = (j >= 0 && j < a.max_entries) ? a.ent[j] : -1;
          if (id < 0 || id >= a.n_ids) {  // cannot happen with a consistent work list
            if (lane == 0) atomicOr(&misc[2], ST_BOUNDS);
            continue;
          }
          const float val = acc[t] * a.bscale[j];
          const size_t o = (size_t)id * a.out_cols;
          if (a.mode == 0) {
            const float up = __shfl_xor_sync(0xffffffffu, val, 1);  // rows 2p (gate) and 2p + 1 (up)
            if (!(lane & 1) && row < a.rows) a.out[o + (row >> 1)] = silu_mul(val, up);
          } else if (row < a.rows) {
            a.out[o + row] = val;
          }
        }
      }
    }
  } else {
    // ---- dequantisation: staged codes -> A K-blocks -------------------------
    const int q = warp & 3, h = (warp - kWarpDeq0) >> 2;
    const int r = 32 * q + lane;
    uint32_t cc = 0, kc = 0, bad = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const TcChunk ch = a.chunks[u / a.tiles];
      const float qmax = ch.bits == 4 ? 15.f : 3.f;
      for (int st = 0; st < nst && ok; ++st, ++cc) {
        const uint32_t cs = cc % kCodeSlots;
        if (!(ok = tc_wait_warp(&full_c[cs], (cc / kCodeSlots) & 1u, abort))) break;
        const uint8_t* cb = sm + kOffCodes + cs * kCodeSlotBytes;
        const int gcount = min(kStageGroups, a.ng - kStageGroups * st);
        // this warp takes the K-blocks kc + j with (kc + j) % 2 == h, all 64
        // inputs of its 32 rows: with an even ring every K slot then has one
        // writer per lane quarter, which keeps the slot parities exact
#pragma unroll 1
        for (int j = h ^ (int)(kc & 1u); j < gcount; j += 2) {
          const uint32_t kj = kc + j, ks = kj % kKSlots;
          if (!(ok = tc_wait_warp(&empty_k[ks], ((kj / kKSlots) & 1u) ^ 1u, abort))) break;
          const uint32_t sbj = *reinterpret_cast<const uint32_t*>(cb + 2 * kHalfBoxBytes + r * 32 + 4 * j);
          const float s = bf16lo(sbj), b = bf16hi(sbj);
          bad |= !(fabsf(s) * qmax + fabsf(b) <= 65504.f);
          const __half2 s2 = __float2half2_rn(s), b2 = __float2half2_rn(b);
          uint32_t v[32];
          if (ch.bits == 4) {
            const uint4 c = *reinterpret_cast<const uint4*>(cb + swz128(r, j));
            const uint4 d = *reinterpret_cast<const uint4*>(cb + kHalfBoxBytes + swz128(r, j));
            const uint32_t w8[8] = {c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint4 o = dequant_word4(w8[i], s2, b2);
              v[4 * i] = o.x; v[4 * i + 1] = o.y; v[4 * i + 2] = o.z; v[4 * i + 3] = o.w;
            }
          } else {
            const uint4 c = *reinterpret_cast<const uint4*>(cb + swz128(r, j));
            const uint32_t w4[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 o0, o1;
              dequant_word2(w4[i], s2, b2, o0, o1);
              v[8 * i] = o0.x; v[8 * i + 1] = o0.y; v[8 * i + 2] = o0.z; v[8 * i + 3] = o0.w;
              v[8 * i + 4] = o1.x; v[8 * i + 5] = o1.y; v[8 * i + 6] = o1.z; v[8 * i + 7] = o1.w;
            }
          }
          tc_fence_after();  // the MMAs that read this slot have completed (empty_k)
          const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + kTmemACol0 + ks * 32;
          tmem_st16(ta, *reinterpret_cast<const uint32_t(*)[16]>(&v[0]));
          tmem_st16(ta + 16, *reinterpret_cast<const uint32_t(*)[16]>(&v[16]));
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&full_a[ks]);
        }
        kc += gcount;
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_c[cs]);
      }
    }
    if (bad) atomicOr(&misc[2], ST_RANGE);
  }

  // ---- teardown: every role has finished or given up --------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
  if (threadIdx.x == 0) {
    const uint32_t st = misc[2] | (*abort ? (uint32_t)ST_TIMEOUT : 0u);
    if (st) atomicOr(&a.hdr->status, st);
  }
}

// ---------------------------------------------------------------------------
// host side: tensor maps and launches
// ---------------------------------------------------------------------------
namespace {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static const EncodeTiled fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiled>(nullptr);
    return reinterpret_cast<EncodeTiled>(p);
  }();
  return fn;
}

// Rows of one weight matrix in every expert of a pool: bytes x rows x experts
// (uint8), box = box_x bytes x kTcM rows x 1 expert.
bool encode_rows(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint64_t depth,
                 uint64_t depth_stride, uint32_t box_x, bool swizzle) {
  const EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {row_bytes, rows, depth};
  const cuuint64_t strides[2] = {row_bytes, depth_stride};
  const cuuint32_t box[3] = {box_x, (cuuint32_t)kTcM, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// B operand rows: fp16 [rows][K], box = 64 inputs x kBBoxRows rows, swizzled.
bool encode_bops(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows) {
  const EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {K, rows};
  const cuuint64_t strides[1] = {K * 2};
  const cuuint32_t box[2] = {64, kBBoxRows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_supported(const TcLaunch& L) {
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (L.H % kGroup || L.I % kGroup || (L.bits != 4 && L.bits != 2)) return false;
  if (L.has_shared && L.shared_bits != 4 && L.shared_bits != 2) return false;
  if (!al16(L.experts) || (L.stride & 15u) || (L.has_shared && !al16(L.shared))) return false;
  return encode_fn() != nullptr;
}

cudaError_t launch_tc_single_item(int B, int* n_uniq, int* uniq_e, int* uniq_off, int* ent, cudaStream_t s) {
  return launch_kernel(tc_single_item_kernel, dim3(1), dim3(256), 0, s, B, n_uniq, uniq_e, uniq_off, ent);
}

cudaError_t launch_tc_plan(const TcPlanArgs& a, cudaStream_t s) {
  return launch_kernel(tc_plan_kernel, dim3(1), dim3(32), 0, s, a);
}

cudaError_t launch_tc_pack(const TcPackArgs& a, int max_entries, cudaStream_t s) {
  if (max_entries <= 0) return cudaSuccess;
  return launch_kernel(tc_pack_kernel, dim3(max_entries), dim3(256), 0, s, a);
}

cudaError_t launch_tc_contract(const TcLaunch& L, int mode, cudaStream_t s) {
  static std::atomic<int> configured[kMaxDevices];
  const Fmt fr = make_fmt(L.bits, L.H, L.I);
  const Fmt fs = make_fmt(L.has_shared ? L.shared_bits : L.bits, L.H, L.I);
  const bool gu = mode == 0;
  const int rows = gu ? 2 * L.I : L.H;
  const int K = gu ? L.H : L.I;
  const uint64_t rb_r = gu ? fr.gu_row : fr.d_row, rb_s = gu ? fs.gu_row : fs.d_row;
  const uint8_t* base_r = L.experts + (gu ? 0 : fr.d_off);
  const uint8_t* base_s = L.has_shared ? L.shared + (gu ? 0 : fs.d_off) : base_r;
  CUtensorMap mc, ms, mcs, mss, mb;
  bool ok = encode_rows(&mc, base_r, rb_r, rows, L.E, L.stride, 128, true) &&
            encode_rows(&ms, base_r, rb_r, rows, L.E, L.stride, 32, false) &&
            encode_rows(&mcs, base_s, rb_s, rows, 1, rb_s * rows, 128, true) &&
            encode_rows(&mss, base_s, rb_s, rows, 1, rb_s * rows, 32, false) &&
            encode_bops(&mb, gu ? L.xops : L.aops, K, 2 * (uint64_t)L.max_entries);
  if (!ok) return cudaErrorInvalidValue;
  TcContractArgs a{};
  a.mode = mode;
  a.rows = rows;
  a.ng = K / kGroup;
  a.tiles = (rows + kTcM - 1) / kTcM;
  a.out_cols = gu ? L.I : L.H;
  a.chunks = L.chunks;
  a.n_chunks = L.n_chunks;
  a.ent = L.ent;
  a.bscale = gu ? L.xscale : L.ascale;
  a.out = gu ? L.a_out : L.d_out;
  a.max_entries = L.max_entries;
  a.n_ids = L.max_entries;
  a.hdr = L.hdr;
  cudaError_t e = ensure_dynamic_smem(tc_contract_kernel, (int)kSmemBytes, configured);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long long max_units = (long long)L.max_chunks * a.tiles;
  const int grid = (int)(max_units < sms ? max_units : sms);
  if (grid <= 0) return cudaSuccess;
  return launch_kernel(tc_contract_kernel, dim3(grid), dim3(kTcThreads), kSmemBytes, s, mc, ms, mcs, mss, mb, a);
}

}  // namespace tc
}  // namespace moe
