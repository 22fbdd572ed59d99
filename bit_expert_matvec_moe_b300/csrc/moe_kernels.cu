// Multi-kernel MoE path (any batch) and the kernels behind moe_pack_weights,
// moe_route and moe_expert_forward.  The single-token layer has its own fused
// kernel (moe_decode_b1.cu); both use the device blocks of moe_device.cuh.
#include "moe_internal.h"

namespace moe {

thread_local bool t_launch_pdl = false;  // see PdlScope

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
  pdl_wait_prior();  // no-op unless launched with programmatic serialisation
  pdl_launch_dependents();
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
// Register-tiled fp32 product over (router rows, tokens, input splits).  A block
// owns kRtRows rows x TOK tokens and one contiguous range of the inputs; each
// thread holds an RT x TT tile of sums.  Stages of kRtK inputs are read into
// registers one stage ahead, then written to shared memory k-major (the rows
// converted from bf16 to fp32 on the way) so that one vector load per operand
// feeds the RT x TT fused multiply-adds of one input.  Every sum runs over its
// inputs in ascending order; the top-K kernel adds the splits' partial sums in
// ascending split order, so results do not depend on scheduling.
constexpr int kRtRows = 64, kRtK = 32, kRtThreads = 256;
constexpr int kRtTargetBlocks = 2 * 148;  // a fixed shape-only target: results do not depend on the device
constexpr int kRtMaxSplits = 32;

static int router_tok_tile(int B) { return B <= 16 ? 16 : (B <= 32 ? 32 : 64); }

int router_splits(int B, int H, int E) {
  const int tiles = ((E + 1 + kRtRows - 1) / kRtRows) * ((B + router_tok_tile(B) - 1) / router_tok_tile(B));
  const int stages = H / kRtK;
  const int want = std::min(std::min(kRtMaxSplits, stages), std::max(1, (kRtTargetBlocks + tiles - 1) / tiles));
  const int per = (stages + want - 1) / want;
  return (stages + per - 1) / per;
}

template <int N>
__device__ __forceinline__ void load_vec(const float* p, float (&v)[N]) {
  static_assert(N == 2 || N == 4, "vector width");
  if constexpr (N == 4) {
    const float4 t = *reinterpret_cast<const float4*>(p);
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  } else {
    const float2 t = *reinterpret_cast<const float2*>(p);
    v[0] = t.x; v[1] = t.y;
  }
}

template <int RT, int TT, int TX>
__global__ void __launch_bounds__(kRtThreads) router_kernel(RouterArgs a) {
  pdl_wait_prior();  // no-op unless launched with programmatic serialisation
  pdl_launch_dependents();
  constexpr int TR = kRtThreads / TX, TOK = TT * TX;
  static_assert(RT * TR == kRtRows, "router row tile");
  constexpr int WSTR = kRtRows + 4, XSTR = TOK + 4;  // k-major strides (16-byte multiples)
  constexpr int WV = kRtRows * kRtK / 8 / kRtThreads;     // 16-byte row pieces per thread
  constexpr int XN = TOK * kRtK / 4;                      // 16-byte token pieces per stage
  constexpr int XV = (XN + kRtThreads - 1) / kRtThreads;
  __shared__ __align__(16) float ws[2][kRtK][WSTR];
  __shared__ __align__(16) float xs[2][kRtK][XSTR];
  const int tid = threadIdx.x;
  const int tx = tid % TX, tr = tid / TX;
  const int nrows = a.E + (a.gate ? 1 : 0);
  const int row0 = blockIdx.x * kRtRows, b0 = blockIdx.y * TOK;
  const int s0 = blockIdx.z * a.stages_per_split, s1 = min(a.H / kRtK, s0 + a.stages_per_split);

  uint4 wr[WV];
  float4 xr[XV];
  auto fetch = [&](int st) {
    const int k0 = st * kRtK;
#pragma unroll
    for (int v = 0; v < WV; ++v) {
      const int i = tid + kRtThreads * v, r = i >> 2, c = i & 3;
      const int row = row0 + r;
      wr[v] = make_uint4(0u, 0u, 0u, 0u);
      if (row < nrows) {
        const uint16_t* R = row < a.E ? a.router + (size_t)row * a.H : a.gate;
        wr[v] = __ldg(reinterpret_cast<const uint4*>(R + k0 + 8 * c));
      }
    }
#pragma unroll
    for (int v = 0; v < XV; ++v) {
      const int i = tid + kRtThreads * v, t = i >> 3, c = i & 7;
      xr[v] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < XN && b0 + t < a.B) xr[v] = *reinterpret_cast<const float4*>(a.xn + (size_t)(b0 + t) * a.H + k0 + 4 * c);
    }
  };
  auto stash = [&](int buf) {
#pragma unroll
    for (int v = 0; v < WV; ++v) {
      const int i = tid + kRtThreads * v, r = i >> 2, c = i & 3;
      const uint32_t w4[4] = {wr[v].x, wr[v].y, wr[v].z, wr[v].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        ws[buf][8 * c + 2 * j][r] = bf16lo(w4[j]);
        ws[buf][8 * c + 2 * j + 1][r] = bf16hi(w4[j]);
      }
    }
#pragma unroll
    for (int v = 0; v < XV; ++v) {
      const int i = tid + kRtThreads * v, t = i >> 3, c = i & 7;
      if (i < XN) {
        xs[buf][4 * c][t] = xr[v].x;
        xs[buf][4 * c + 1][t] = xr[v].y;
        xs[buf][4 * c + 2][t] = xr[v].z;
        xs[buf][4 * c + 3][t] = xr[v].w;
      }
    }
  };

  float acc[RT][TT];
#pragma unroll
  for (int i = 0; i < RT; ++i)
#pragma unroll
    for (int j = 0; j < TT; ++j) acc[i][j] = 0.f;
  if (s0 < s1) {
    fetch(s0);
    stash(0);
  }
  __syncthreads();
  for (int st = s0; st < s1; ++st) {
    const int buf = (st - s0) & 1;
    if (st + 1 < s1) fetch(st + 1);
#pragma unroll 8
    for (int k = 0; k < kRtK; ++k) {
      float w[RT], x[TT];
      load_vec<RT>(&ws[buf][k][tr * RT], w);
      load_vec<TT>(&xs[buf][k][tx * TT], x);
#pragma unroll
      for (int i = 0; i < RT; ++i)
#pragma unroll
        for (int j = 0; j < TT; ++j) acc[i][j] = fmaf(w[i], x[j], acc[i][j]);
    }
    if (st + 1 < s1) stash(buf ^ 1);
    __syncthreads();
  }
  // partial sums of this split: logits[split][token][row]
  float* out = a.logits + (size_t)blockIdx.z * a.B * (a.E + 1);
#pragma unroll
  for (int j = 0; j < TT; ++j) {
    const int b = b0 + tx * TT + j;
    if (b >= a.B) continue;
#pragma unroll
    for (int i = 0; i < RT; ++i) {
      const int row = row0 + tr * RT + i;
      if (row < nrows) out[(size_t)b * (a.E + 1) + row] = acc[i][j];
    }
  }
}

// ---------------------------------------------------------------------------
// softmax / top-K / renormalise per token: one warp per token
// ---------------------------------------------------------------------------
constexpr int kTopkPer = 32;  // experts per lane: up to 1024 experts
constexpr int kTopkThreads = 512;  // one logit per thread up to 512 experts
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(TopkArgs a) {
  pdl_wait_prior();  // no-op unless launched with programmatic serialisation
  pdl_launch_dependents();
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  // logits of this token: the router's split partial sums added in split order,
  // then the caller's offset (routed experts only)
  __shared__ float s_lg[kTopkPer * 32 + 1];
  const size_t pstride = (size_t)a.B * (a.E + 1);
  const float* part = a.logits + (size_t)b * (a.E + 1);
  const int nrows = a.E + (a.has_gate ? 1 : 0);
  for (int e = tid; e < nrows; e += blockDim.x) {
    float v = part[e];
    int sp = 1;
    for (; sp + 16 <= a.splits; sp += 16) {  // sixteen loads in flight, added in split order
      float p[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) p[i] = part[(size_t)(sp + i) * pstride + e];
#pragma unroll
      for (int i = 0; i < 16; ++i) v += p[i];
    }
    for (; sp < a.splits; ++sp) v += part[(size_t)sp * pstride + e];
    if (e < a.E && a.offset) v += a.offset[(size_t)b * a.E + e];
    s_lg[e] = v;
  }
  __syncthreads();
  if (tid >= 32) return;
  const float* lg = s_lg;
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
// token -> expert grouping (one block).  Work items: first the shared expert,
// when present, in items of at most kSharedChunk tokens (slot K of every token:
// the heaviest items, so they are dispatched first and spread over more
// blocks), then every touched routed expert once, ascending by id, with its
// (token, slot) entries ascending by token.  Item u covers entries
// [uniq_off[u], uniq_off[u + 1]); expert id -1 is the shared expert.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kBlock) bucket_kernel(BucketArgs a) {
  pdl_wait_prior();  // no-op unless launched with programmatic serialisation
  pdl_launch_dependents();
  extern __shared__ int bk_smem[];
  const int n = a.B * a.K;
  int* cnt = bk_smem;     // [E]
  int* off = cnt + a.E;   // [E]
  int* ids = off + a.E;   // [n] the routing choices, staged
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) cnt[e] = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) ids[i] = a.idx[i];
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) atomicAdd(&cnt[ids[i]], 1);
  __syncthreads();
  // thread t owns experts 2t and 2t + 1: one block-wide exclusive scan of
  // (entries, touched experts) in expert order gives every expert's first
  // entry and its work-item number
  __shared__ int s_wsum[2][kWarps];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int e0 = 2 * tid, e1 = 2 * tid + 1;
  const int c0 = e0 < a.E ? cnt[e0] : 0, c1 = e1 < a.E ? cnt[e1] : 0;
  const int f0 = c0 > 0, f1 = c1 > 0;
  int ic = c0 + c1, iu = f0 + f1;  // inclusive scans within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int vc = __shfl_up_sync(0xffffffffu, ic, o), vu = __shfl_up_sync(0xffffffffu, iu, o);
    if (lane >= o) { ic += vc; iu += vu; }
  }
  if (lane == 31) { s_wsum[0][wid] = ic; s_wsum[1][wid] = iu; }
  __syncthreads();
  int wc = 0, wu = 0;  // totals of the earlier warps
  for (int w = 0; w < wid; ++w) { wc += s_wsum[0][w]; wu += s_wsum[1][w]; }
  const int n_shared_items = a.has_shared ? (a.B + kSharedChunk - 1) / kSharedChunk : 0;
  const int base = a.has_shared ? a.B : 0;  // the shared expert's entries come first
  const int xc = base + wc + ic - (c0 + c1), xu = n_shared_items + wu + iu - (f0 + f1);
  if (e0 < a.E) {
    off[e0] = xc;
    if (f0) { a.uniq_e[xu] = e0; a.uniq_off[xu] = xc; }
  }
  if (e1 < a.E) {
    off[e1] = xc + c0;
    if (f1) { a.uniq_e[xu + f0] = e1; a.uniq_off[xu + f0] = xc + c0; }
  }
  if (tid < n_shared_items) {
    a.uniq_e[tid] = -1;
    a.uniq_off[tid] = tid * kSharedChunk;
  }
  if (tid == blockDim.x - 1) {  // the last thread's inclusive totals are the block's
    a.uniq_off[xu + f0 + f1] = xc + c0 + c1;
    *a.n_uniq = xu + f0 + f1;
  }
  __syncthreads();
  // entry i = (b, k): its position among entries of the same expert is the
  // number of earlier entries (in (b, k) order) with that expert
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int e = ids[i];
    int pos = 0;
    for (int j = 0; j < i; ++j) pos += (ids[j] == e);
    const int b = i / a.K, k = i % a.K;
    a.ent[off[e] + pos] = b * a.nslots + k;
  }
  if (a.has_shared)
    for (int b = threadIdx.x; b < a.B; b += blockDim.x) a.ent[b] = b * a.nslots + a.K;
}

// ---------------------------------------------------------------------------
// weight-stationary grouped matvecs (B > 1)
// ---------------------------------------------------------------------------
// A block stages a tile of one expert's rows in shared memory once (cp.async),
// then applies every token routed to that expert.  Lane g of a warp owns group
// g of its row chunk: it loads the token's limbs of that group once (registers)
// and runs them against each of the warp's rows of the tile (codes from shared
// memory, conflict-free 16-byte loads in the packed layout); the lanes of a row
// are reduced by shuffles.  Tokens go kTok at a time between block barriers;
// per-row partials (one per row chunk) are summed in a fixed order, so results
// are deterministic.  grid = (row tiles, work items); item u is expert
// uniq_e[u] (or the shared expert) with its token entries; without a list
// (single-expert mode) the item is `blob` with tokens 0..B-1.
constexpr int kWsThreads = 256;
constexpr int kWsWarps = kWsThreads / 32;
constexpr int kGuTile = 32;   // gate/up rows per tile at most (16 pairs)
constexpr int kDnTile = 128;  // down rows per tile at most
constexpr int kTok = 8;       // tokens between block barriers
constexpr int kMaxRowsPerLane = 8;

// rows of a tile: what the warps' lane streams cover with kMaxRowsPerLane rows
// per lane (rows of ng groups), capped; gate/up tiles hold whole row pairs
__host__ __device__ inline int tile_cover(int ng) {
  const RowMap m = make_rowmap(ng);
  return kMaxRowsPerLane * (kWsWarps / m.chunks) * m.rpp;
}
__host__ __device__ inline int gu_tile_rows(int H) { return min(kGuTile, tile_cover(H / kGroup)) & ~1; }
__host__ __device__ inline int dn_tile_rows(int I) { return min(kDnTile, tile_cover(I / kGroup)); }

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}

// rows [0, nrows) (row r at src(r), row_bytes each, a multiple of 16) to dst + r * row_bytes
template <typename Src>
__device__ __forceinline__ void stage_rows(uint8_t* dst, Src src, int nrows, int row_bytes) {
  const int chunks = row_bytes / 16;
  for (int i = threadIdx.x; i < nrows * chunks; i += blockDim.x) {
    const int r = i / chunks, c = i - r * chunks;
    cp_async16(dst + (size_t)r * row_bytes + 16 * c, src(r) + 16 * c);
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
}

// partial dots of one token with the warp's rows of a staged tile: rows
// r_first + k * r_step (k < kRows, those < nrows), row r at tile + r * row_bytes;
// out[k] = the row's sum over this lane's chunk of groups (same on all lanes of
// the row).  All lanes of the warp call it.
template <int BITS, int kRows>
__device__ __forceinline__ void tile_rows(const uint8_t* tile, int row_bytes, int codes_bytes, int ng, int g,
                                          bool gact, const Limbs& L, float2 es, int r_first, int r_step, int nrows,
                                          int lpr, float (&out)[kRows]) {
  float v[kRows];
#pragma unroll
  for (int k = 0; k < kRows; ++k) {
    const int r = r_first + k * r_step;
    v[k] = (gact && r < nrows) ? row_group<BITS>(tile + (size_t)r * row_bytes, ng, codes_bytes, g, L, es) : 0.f;
  }
#pragma unroll
  for (int k = 0; k < kRows; ++k) out[k] = row_reduce(v[k], lpr);
}

// One work item's tile: rows [0, nrows) of the tile staged; per token chunk,
// warp w takes chunk w % chunks of the groups and rows (w / chunks) * rpp + ...;
// the partials go to part[t][r][chunk] and finish(t0, ntok) combines them.
template <int BITS, int kRows, typename Vec, typename Finish>
__device__ __forceinline__ void tile_tokens(const uint8_t* tile, int row_bytes, int codes_bytes, int ng, int nrows,
                                            int nent, Vec vec_of, float* part, Finish finish) {
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  const RowMap m = make_rowmap(ng);
  const int chunk = wi % m.chunks, nstreams = kWsWarps / m.chunks;
  const int g = chunk * 32 + lane % m.lpr;
  const bool gact = g < ng && wi < nstreams * m.chunks;
  const int r_first = (wi / m.chunks) * m.rpp + lane / m.lpr, r_step = nstreams * m.rpp;
  for (int t0 = 0; t0 < nent; t0 += kTok) {
    const int ntok = min(kTok, nent - t0);
    for (int t = 0; t < ntok; ++t) {
      const uint8_t* q;
      const float2* e;
      vec_of(t0 + t, q, e);
      Limbs L;
      float2 es = make_float2(0.f, 0.f);
      if (gact) {
        load_limbs(q, ng, g, L);
        es = e[g];
      } else {
        zero_limbs(L);
      }
      float o[kRows];
      tile_rows<BITS, kRows>(tile, row_bytes, codes_bytes, ng, g, gact, L, es, r_first, r_step, nrows, m.lpr, o);
      if (lane % m.lpr == 0 && gact) {
#pragma unroll
        for (int k = 0; k < kRows; ++k) {
          const int r = r_first + k * r_step;
          if (r < nrows) part[(t * nrows + r) * m.chunks + chunk] = o[k];
        }
      }
    }
    __syncthreads();
    finish(t0, ntok, m.chunks);
    __syncthreads();
  }
}

template <int BITS>
__device__ void gateup_tile(const GateUpArgs& a, const uint8_t* blob, const Fmt& f, const int* ent, int nent,
                            uint8_t* sm) {
  const int tile = gu_tile_rows(f.H);
  const int p0 = blockIdx.x * (tile / 2);  // first gate/up row pair of the tile
  const int npair = min(tile / 2, f.I - p0);
  if (npair <= 0) return;
  const int nrows = 2 * npair;
  // tile row r: pair r / 2, gate row for even r, up row for odd r (the blob's order)
  stage_rows(sm, [&](int r) { return blob + (size_t)(p0 + (r >> 1)) * f.gu_pair + (size_t)(r & 1) * f.gu_row; },
             nrows, f.gu_row);
  float* part = reinterpret_cast<float*>(sm + (size_t)tile * f.gu_row);  // [kTok][rows][chunks]
  auto entry = [&](int t) { return ent ? ent[t] : t * a.nslots; };       // b * nslots + slot
  auto vec_of = [&](int t, const uint8_t*& q, const float2*& e) {
    const int b = entry(t) / a.nslots;
    q = a.xq + (size_t)b * f.ng_h * kLimbBytes;
    e = a.xe + (size_t)b * f.ng_h;
  };
  auto finish = [&](int t0, int ntok, int chunks) {
    for (int j = threadIdx.x; j < ntok * npair; j += blockDim.x) {
      const int t = j / npair, pp = j - t * npair;
      float g = 0.f, u = 0.f;
      for (int c = 0; c < chunks; ++c) {
        g += part[(t * nrows + 2 * pp) * chunks + c];
        u += part[(t * nrows + 2 * pp + 1) * chunks + c];
      }
      a.a_out[(size_t)entry(t0 + t) * f.I + p0 + pp] = silu_mul(g, u);
    }
  };
  tile_tokens<BITS, kMaxRowsPerLane>(sm, f.gu_row, f.gu_codes, f.ng_h, nrows, nent, vec_of, part, finish);
}

__global__ void __launch_bounds__(kWsThreads, 2) gateup_kernel(GateUpArgs a) {
  pdl_wait_prior();  // no-op unless launched with programmatic serialisation
  pdl_launch_dependents();
  extern __shared__ __align__(16) uint8_t sm[];
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
    gateup_tile<4>(a, blob, f, ent, nent, sm);
  else
    gateup_tile<2>(a, blob, f, ent, nent, sm);
}

template <int BITS>
__device__ void down_tile(const DownArgs& a, const uint8_t* blob, const Fmt& f, const int* ent, int nent, uint8_t* sm) {
  const int tile = dn_tile_rows(f.I);
  const int j0 = blockIdx.x * tile;
  const int nrows = min(tile, f.H - j0);
  if (nrows <= 0) return;
  stage_rows(sm, [&](int r) { return blob + f.d_off + (size_t)(j0 + r) * f.d_row; }, nrows, f.d_row);
  float* part = reinterpret_cast<float*>(sm + (size_t)tile * f.d_row);  // [kTok][rows][chunks]
  auto entry = [&](int t) { return ent ? ent[t] : t * a.nslots; };
  auto vec_of = [&](int t, const uint8_t*& q, const float2*& e) {
    const int en = entry(t);
    q = a.aq + (size_t)en * f.ng_i * kLimbBytes;
    e = a.ae + (size_t)en * f.ng_i;
  };
  auto finish = [&](int t0, int ntok, int chunks) {
    for (int j = threadIdx.x; j < ntok * nrows; j += blockDim.x) {
      const int t = j / nrows, r = j - t * nrows;
      float sum = 0.f;
      for (int c = 0; c < chunks; ++c) sum += part[(t * nrows + r) * chunks + c];
      a.d_out[(size_t)entry(t0 + t) * f.H + j0 + r] = sum;
    }
  };
  tile_tokens<BITS, kMaxRowsPerLane>(sm, f.d_row, f.d_codes, f.ng_i, nrows, nent, vec_of, part, finish);
}

__global__ void __launch_bounds__(kWsThreads, 2) down_kernel(DownArgs a) {
  pdl_wait_prior();  // no-op unless launched with programmatic serialisation
  pdl_launch_dependents();
  extern __shared__ __align__(16) uint8_t sm[];
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
    down_tile<4>(a, blob, f, ent, nent, sm);
  else
    down_tile<2>(a, blob, f, ent, nent, sm);
}

// ---------------------------------------------------------------------------
// combine: h[b] += sum_k w[b][k] d[b][k] + gs[b] d[b][K]   (fixed order), or
// the single-expert output out[b] = (acc ? out[b] : 0) + row_w[b] d[b][0]
// ---------------------------------------------------------------------------
__global__ void combine_kernel(CombineArgs a) {
  pdl_wait_prior();  // no-op unless launched with programmatic serialisation
  pdl_launch_dependents();
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
  return launch_kernel(norm_quant_kernel, dim3(B), dim3(kBlock), sm, s, a);
}
cudaError_t launch_router(const RouterArgs& a, cudaStream_t s) {
  const int rows = a.E + (a.gate ? 1 : 0);
  const int tok = router_tok_tile(a.B);
  const int splits = (a.H / kRtK + a.stages_per_split - 1) / a.stages_per_split;
  if (a.stages_per_split < 1 || splits != router_splits(a.B, a.H, a.E)) return cudaErrorInvalidValue;
  dim3 grid((rows + kRtRows - 1) / kRtRows, (a.B + tok - 1) / tok, splits);
  if (tok == 16)
    return launch_kernel(router_kernel<2, 2, 8>, grid, dim3(kRtThreads), 0, s, a);
  else if (tok == 32)
    return launch_kernel(router_kernel<4, 2, 16>, grid, dim3(kRtThreads), 0, s, a);
  else
    return launch_kernel(router_kernel<4, 4, 16>, grid, dim3(kRtThreads), 0, s, a);
}
int router_stages_per_split(int B, int H, int E) {
  const int stages = H / kRtK, sp = router_splits(B, H, E);
  return (stages + sp - 1) / sp;
}
cudaError_t launch_topk(const TopkArgs& a, int B, cudaStream_t s) {
  return launch_kernel(topk_kernel, dim3(B), dim3(kTopkThreads), 0, s, a);
}
cudaError_t launch_bucket(const BucketArgs& a, cudaStream_t s) {
  const size_t sm = (size_t)(2 * a.E + a.B * a.K) * sizeof(int);
  if (sm > 48 * 1024 || a.E > 2 * kBlock) return cudaErrorInvalidValue;  // two experts per thread
  return launch_kernel(bucket_kernel, dim3(1), dim3(kBlock), sm, s, a);
}
// shared memory of one weight-stationary tile: staged rows and the partials of
// one token chunk ([kTok][rows][row chunks]); sized for the wider code width
static size_t tile_smem(int rows, int row_bytes_4, int row_bytes_2, int ng) {
  return (size_t)rows * std::max(row_bytes_4, row_bytes_2) + (size_t)kTok * rows * ((ng + 31) / 32) * 4;
}
cudaError_t launch_gateup(const GateUpArgs& a, int items, cudaStream_t s) {
  const int tile = gu_tile_rows(a.H);
  if (tile < 2) return cudaErrorInvalidValue;
  const size_t sm = tile_smem(tile, make_fmt(4, a.H, a.I).gu_row, make_fmt(2, a.H, a.I).gu_row, a.H / kGroup);
  static std::atomic<int> configured[kMaxDevices];
  const cudaError_t e = ensure_dynamic_smem(gateup_kernel, (int)sm, configured);
  if (e != cudaSuccess) return e;
  dim3 grid((a.I + tile / 2 - 1) / (tile / 2), items);
  return launch_kernel(gateup_kernel, grid, dim3(kWsThreads), sm, s, a);
}
cudaError_t launch_down(const DownArgs& a, int items, cudaStream_t s) {
  const int tile = dn_tile_rows(a.I);
  if (tile < 1) return cudaErrorInvalidValue;
  const size_t sm = tile_smem(tile, make_fmt(4, a.H, a.I).d_row, make_fmt(2, a.H, a.I).d_row, a.I / kGroup);
  static std::atomic<int> configured[kMaxDevices];
  const cudaError_t e = ensure_dynamic_smem(down_kernel, (int)sm, configured);
  if (e != cudaSuccess) return e;
  dim3 grid((a.H + tile - 1) / tile, items);
  return launch_kernel(down_kernel, grid, dim3(kWsThreads), sm, s, a);
}
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) {
  const size_t n = (size_t)a.B * a.H;
  const int grid = (int)std::min<size_t>((n + 255) / 256, 148 * 8);
  return launch_kernel(combine_kernel, grid, dim3(256), 0, s, a);
}

}  // namespace moe
