// Single-token MoE layer in one launch of one block per SM.
//
// Block c of P owns gate/up row pairs [c*I/P, (c+1)*I/P) and down rows
// [c*H/P, (c+1)*H/P) of every expert the token uses, and router rows
// [c*E/P, (c+1)*E/P).  Its weight bytes arrive by bulk copies (TMA engine)
// into shared memory, each with its own mbarrier:
//   start           h, router rows, shared expert gate/up rows and down rows
//   after top-K     gate/up rows of all K routed experts (they fit side by side)
//   after gate/up k down rows of routed expert k (once its gate/up rows landed)
// Grid-wide data dependencies go through the workspace: every published word
// carries its layer's epoch in its upper half (one epoch per layer, so one per
// launch of this kernel; a reader sees either the old word or the new one,
// never a mix, and polls a word again until its epoch is the current layer's).  The logits are polled directly; for the activations, which
// every block reads in full, one relaxed counter tells a reader when every
// block has published, and late words are polled again after it.
// Phases of a block:
//   h -> h*gamma and a block sum for the RMS factor r
//   router rows -> published logits
//   limbs of h*gamma (r multiplies each gate/up dot product instead, so the
//        limbs do not wait for the norm; quantised once the logits are out)
//   warps 1..: shared expert gate/up.  Meanwhile warp 0: poll every block's
//           logits (16 words per lane in flight); top-K (every block, same
//           result); issue the routed gate/up copies whose slots do not
//           overlap the shared slice; softmax over the chosen; then its own
//           shared rows and, once every warp is done with the shared slice,
//           the remaining copies
//   routed gate/up rows expert by expert as their copies land
//   SwiGLU of every expert's rows, times its routing weight -> published
//   wait for the activation counter; every thread loads its 12 words straight
//   from the workspace (late ones polled together); limbs of each 64-group
//   down rows of every expert as one long dot product per row -> h[rows] += y
// Routing never leaves the device.  Every wait is bounded (1 s): on timeout the
// block records MOE_ERR_TIMEOUT, waits (bounded) for its own copies in flight,
// advances the counters it still owes and leaves; later launches on the same
// workspace return at once until the status word is read.  Nothing lives in
// local memory: with ~227 KB of shared memory per block the L1 cache is small,
// and spilled state would go to L2.
//
// Limits of this kernel (the host falls back to the multi-kernel path outside
// them): hidden <= 4096, inter <= 2048, experts <= 1024, top-K <= 8, and the
// plan must fit in shared memory.
//
// With programmatic dependent launch (kPDL) the router rows are copied before
// griddepcontrol.wait, i.e. while the previous kernel on the stream may still
// run; nothing the caller writes (h, offsets, workspace) is read before that
// wait.
//
// decode_stack_kernel runs the layers of one token in one launch, the same
// phases once per layer.  Layer l's output rows are published like the
// activations (epoch words, one relaxed counter) and read back by every block
// as layer l + 1's input; each block keeps its own rows in registers for the
// residual.  The next layer's router rows and shared gate/up rows are copied
// as soon as the routed gate/up slices are dead (after the gate/up phase), and
// its shared down rows once the down rows are done, so that they have landed
// when the layer starts.  The layers' epochs are consecutive; every mbarrier
// completes one phase per copy, its parity tracked per layer.
#include <type_traits>

#include "moe_internal.h"

namespace moe {

namespace {

__device__ __forceinline__ int lo_row(int c, int P, int n) { return (int)((long long)c * n / P); }

// Phase stamps (globaltimer) of every block, in builds with MOE_TIMELINE only.
#ifdef MOE_TIMELINE
constexpr int kStamps = 32;
__device__ unsigned long long g_timeline[1024 * kStamps];
#define STAMP(i) (g_timeline[blockIdx.x * kStamps + (i)] = globaltimer())
#else
#define STAMP(i) ((void)0)
#endif

// Slot of activation value i in its expert's published vector: inside each
// group of 64, value 4j + t goes to slot 16t + j, so that the half-warp that
// reads a group (lane j takes values 4j .. 4j+3) reads 16 consecutive words per
// load.
__device__ __forceinline__ int act_slot(int i) { return (i & ~63) | ((i & 3) << 4) | ((i >> 2) & 15); }

// Slot of output row j in a stack launch's published h: inside each chunk of
// 128, value 4l + t goes to slot 32t + l, so that the warp that reads a chunk
// (lane l takes values 4l .. 4l+3) reads 32 consecutive words per load.  The
// published vector spans H rounded up to 128 words.
__device__ __forceinline__ int h_slot(int j) { return (j & ~127) | ((j & 3) << 5) | ((j >> 2) & 31); }

constexpr int kDnRows = 5;  // down rows per thread (the plan checks rows_d <= kDnRows * sets)

// Limbs of kG groups of 64 values, each held four per lane by a half-warp
// (lane j of the half holds values 4j .. 4j+3 of its group); all 32 lanes of
// the warp must call it.  The kG groups are independent, so their shuffle
// chains interleave.  Each lane assembles three limb words per group; when
// store[k], it writes them (limb vector vec[k] of ng groups, group g[k]) and
// lane 0 of the half writes the group factors, times scale[k], to *es[k]
// (scaling both factors scales the group's values).  Returns false when a
// value is not finite.
//
// Per group: E is the exponent of the largest |value| (max = f * 2^E, f in
// [0.5, 1)), read from its bits; every value becomes the integer
// round(v * 2^(22 - E)) (|X| < 2^22), rounded to nearest-even by adding and
// removing 1.5 * 2^23 in fp32, which is exact in that range.
template <int kG>
__device__ __forceinline__ bool quantize_groups(const float4 (&x)[kG], int lane, const bool (&store)[kG],
                                                uint8_t* const (&vec)[kG], int ng, const int (&g)[kG],
                                                float2* const (&es)[kG], const float (&scale)[kG]) {
  const int j = lane & 15;
  float m[kG];
#pragma unroll
  for (int k = 0; k < kG; ++k) m[k] = fmaxf(fmaxf(fabsf(x[k].x), fabsf(x[k].y)), fmaxf(fabsf(x[k].z), fabsf(x[k].w)));
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) {
#pragma unroll
    for (int k = 0; k < kG; ++k) m[k] = fmaxf(m[k], __shfl_xor_sync(0xffffffffu, m[k], o));
  }
  bool finite_all = true;
  int X[kG][4], s[kG];
  float dn[kG];
#pragma unroll
  for (int k = 0; k < kG; ++k) {
    const bool finite = isfinite(m[k]);
    finite_all &= finite;
    const int e = (int)((__float_as_uint(m[k]) >> 23) & 255u);
    const int E = (m[k] > 0.f && finite) ? max(e - 126, -100) : 0;
    const float up = __uint_as_float((uint32_t)(127 + 22 - E) << 23);  // 2^(22-E)
    dn[k] = __uint_as_float((uint32_t)(127 - 22 + E) << 23);           // 2^(E-22)
    const float v[4] = {x[k].x, x[k].y, x[k].z, x[k].w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      X[k][i] = finite ? __float_as_int(fmaf(v[i], up, 12582912.0f)) - 0x4B400000 : 0;
    s[k] = X[k][0] + X[k][1] + X[k][2] + X[k][3];
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) {
#pragma unroll
    for (int k = 0; k < kG; ++k) s[k] += __shfl_xor_sync(0xffffffffu, s[k], o);
  }
  // word q = j >> 1 holds values 8q .. 8q+7; lane 2q has 8q..8q+3, lane 2q+1
  // has 8q+4..8q+7.  The even lane builds the "even" limb words (values 8q,
  // 8q+2, 8q+4, 8q+6), the odd lane the "odd" ones (8q+1, 8q+3, 8q+5, 8q+7).
  const bool odd = j & 1;
  const int q = j >> 1;
#pragma unroll
  for (int k = 0; k < kG; ++k) {
    const int gotA = __shfl_xor_sync(0xffffffffu, odd ? X[k][0] : X[k][1], 1);
    const int gotB = __shfl_xor_sync(0xffffffffu, odd ? X[k][2] : X[k][3], 1);
    const int v0 = odd ? gotA : X[k][0], v1 = odd ? gotB : X[k][2], v2 = odd ? X[k][1] : gotA,
              v3 = odd ? X[k][3] : gotB;
    if (store[k]) {
#pragma unroll
      for (int l = 0; l < 3; ++l) {
        const uint32_t word = ((uint32_t)(v0 >> (8 * l)) & 255u) | (((uint32_t)(v1 >> (8 * l)) & 255u) << 8) |
                              (((uint32_t)(v2 >> (8 * l)) & 255u) << 16) | (((uint32_t)(v3 >> (8 * l)) & 255u) << 24);
        const int w = 6 * q + 2 * l + (odd ? 1 : 0);
        *reinterpret_cast<uint32_t*>(vec[k] + ((size_t)(w >> 2) * ng + g[k]) * 16 + (w & 3) * 4) = word;
      }
      if (j == 0) *es[k] = make_float2(dn[k] * scale[k], (float)s[k] * dn[k] * scale[k]);
    }
  }
  return finite_all;
}

// Dot products of one lane's group with up to two rows of a slice in shared
// memory (rows r_first and r_first + step, those < nrows).  Row r starts at
// base + (r >> 1) * 2 * stride + (r & 1) * stride for gate/up pairs, or
// base + r * stride for down rows.  The lpr lanes of a row are reduced; every
// lane of the row gets the row's partial over its chunk of groups.
template <int BITS, bool kPairs>
__device__ __forceinline__ void slice_rows2(const uint8_t* base, int stride, int codes, int ng, int g, bool gact,
                                            const Limbs& L, float2 es, int r_first, int step, int nrows, int lpr,
                                            float& out0, float& out1) {
  float v[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int r = r_first + k * step;
    v[k] = 0.f;
    if (gact && r < nrows) {
      const uint8_t* row = kPairs ? base + (size_t)(r >> 1) * (2 * stride) + (size_t)(r & 1) * stride
                                  : base + (size_t)r * stride;
      v[k] = row_group<BITS>(row, ng, codes, g, L, es);
    }
  }
  out0 = row_reduce(v[0], lpr);
  out1 = row_reduce(v[1], lpr);
}

}  // namespace

// The body of both kernels for layer l: the only layer (decode_b1_kernel), or
// layer l of one token's layers (decode_stack_kernel, which calls it for
// l = 0, 1, ...: layer l's output rows are published for every block and read
// back as layer l + 1's input; the next layer's router rows and shared gate/up
// rows are copied once the routed gate/up slices are dead, its shared down rows
// once the down rows are done).  Every layer has its own epoch, one above the
// previous layer's.  The launch prologue runs with layer 0.  Returns false
// when the block gave up (the launch is then over for it).
template <bool kPDL, int kRB, int kSB, bool kStack>
__device__ __forceinline__ bool decode_body(const DecodeArgs& a, const DecodeLayer* layers, int nlayers,
                                            unsigned long long* pub_h, int l) {
  // every piece of block scratch lives in the planned dynamic region, whose
  // base is rounded up here to 128 bytes (the plan reserves the slack)
  extern __shared__ uint8_t sm_raw[];
  uint8_t* const sm = sm_raw + ((128u - (uint32_t)(__cvta_generic_to_shared(sm_raw) & 127u)) & 127u);

  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int P = gridDim.x, c = blockIdx.x;
  const int H = a.H, I = a.I, E = a.E, K = a.K, hs = a.has_shared;
  const int NE = K + hs;
  const int ngh = H / kGroup, ngi = I / kGroup;
  const int r0 = lo_row(c, P, I), nr = lo_row(c + 1, P, I) - r0;
  const int j0 = lo_row(c, P, H), nj = lo_row(c + 1, P, H) - j0;
  const int e0 = lo_row(c, P, E), ne = lo_row(c + 1, P, E) - e0;
  const int nrr = ne + ((a.has_gate && c == 0) ? 1 : 0);  // router rows of this block

  // formats by value (4-bit and 2-bit), so that no per-expert choice needs memory
  const Fmt f4 = make_fmt(4, H, I), f2 = make_fmt(2, H, I);
  // code widths are template arguments (routed kRB, shared kSB): each
  // instantiation holds only the unpacking code it runs, which keeps the
  // kernel's instruction footprint down
  const int s_gu_pair = kSB == 4 ? f4.gu_pair : f2.gu_pair;
  const int s_d_row = kSB == 4 ? f4.d_row : f2.d_row;
  const size_t s_d_off = kSB == 4 ? f4.d_off : f2.d_off;
  const int r_gu_pair = kRB == 4 ? f4.gu_pair : f2.gu_pair;
  const int r_d_row = kRB == 4 ? f4.d_row : f2.d_row;
  const size_t r_d_off = kRB == 4 ? f4.d_off : f2.d_off;

  uint8_t* const G = sm + a.plan.off_g;
  uint8_t* const D = sm + a.plan.off_dn;
  uint8_t* const AL = sm + a.plan.off_al;  // limbs: of x first, then of every weighted a
  float2* const AE = reinterpret_cast<float2*>(sm + a.plan.off_ae);
  float* const part = reinterpret_cast<float*>(sm + a.plan.off_part);    // [NE][part_stride]
  float* const rpart = reinterpret_cast<float*>(sm + a.plan.off_rpart);  // [rows_r][kWarps]
  float* const ysm = reinterpret_cast<float*>(sm + a.plan.off_y);        // [rows_d]
  float* const pdn = reinterpret_cast<float*>(G + a.plan.off_pdn);  // down partials [rows_d][NE * ngi]
  uint64_t* const bar = reinterpret_cast<uint64_t*>(sm + a.plan.off_bar);
  float* const s_red = reinterpret_cast<float*>(sm + a.plan.off_misc);               // [kWarps]
  int* const s_idx = reinterpret_cast<int*>(sm + a.plan.off_misc + 64);              // [kMaxTopK]
  float* const s_val = reinterpret_cast<float*>(sm + a.plan.off_misc + 96);          // [kMaxTopK]
  float* const s_coef = reinterpret_cast<float*>(sm + a.plan.off_misc + 128);        // [kMaxTopK + 1]
  // issued, failed, epoch, hook, bumped, act wait, issued for the next layer,
  // h wait, barrier phases (bit i: the parity of barrier i's phase in this
  // layer; written by thread 0 at the start of a layer, always 0 for one layer)
  uint32_t* const s_mask = reinterpret_cast<uint32_t*>(sm + a.plan.off_misc + 168);
  // (stack) the output-row counter as this launch found it
  unsigned long long* const s_hbase = reinterpret_cast<unsigned long long*>(sm + a.plan.off_misc + 208);
  // the current layer's pointers: the launch argument, or (stack) a copy in
  // shared memory made at the start of each layer, followed by the next
  // layer's (read by the thread that issues its early copies)
  DecodeLayer* const s_ly = reinterpret_cast<DecodeLayer*>(sm + a.plan.off_misc + 256);
  // (stack) the block's rows of the layer's input, for the residual: warp 0's
  // lanes write and read their own entries
  float* const s_hres = reinterpret_cast<float*>(sm + a.plan.off_misc + 256 + 2 * sizeof(DecodeLayer));
  auto ly = [&]() -> const DecodeLayer& {
    if constexpr (kStack)
      return *s_ly;
    else
      return a.ly;
  };
  // layers l and l + 1 (when there is one) into s_ly[0], s_ly[1]: threads
  // 0..17; read after the next block barrier
  auto copy_layer = [&](int l) {
    constexpr int kWords = (int)(sizeof(DecodeLayer) / 8);
    if (tid < (l + 1 < nlayers ? 2 : 1) * kWords)
      reinterpret_cast<unsigned long long*>(s_ly)[tid] = reinterpret_cast<const unsigned long long*>(layers + l)[tid];
  };
  // the thread that issues the next layer's early copies: one with no SwiGLU
  // rows (at most 9 experts x 32 rows per block) that sums a down row only in
  // blocks with more than 30 of them
  constexpr int kPrefetchTid = kBlock - 32;
  const size_t gu_slot = a.plan.gu_slot, dn_slot = a.plan.dn_slot;
  const int part_stride = a.plan.part_stride;
  // mbarriers: [0] router rows, [1 + p] gate/up of expert p, [1 + NE + p] down
  // of expert p (expert p = 0 is the shared expert when present), then h.
  // Each completes one phase per copy.
  const int bar_h = 1 + 2 * NE, nbar = bar_h + 1;
  auto parity = [&](int i) -> uint32_t {
    if constexpr (kStack)
      return (*(volatile uint32_t*)&s_mask[8] >> i) & 1u;
    else
      return 0u;
  };
  float hres = 0.f;    // h[j0 + tid] of the layer's input (threads < nj; one layer)
  float* const hbuf = reinterpret_cast<float*>(G + a.plan.off_hbuf);

  // ---- prologue.
  // Every block reads all of h (one bulk copy), the logits and the
  // activations (polled words).
  // Barrier set-up, visible to every thread and to the copy engine before the
  // first copy is issued:
  if (l == 0) {
    if (tid == 0) {
      STAMP(0);
      for (int i = 0; i < nbar; ++i) mbar_init(&bar[i], 1);
      fence_mbar_init();
      fence_proxy_async();
      s_mask[0] = 0u;
      s_mask[1] = 0u;
      s_mask[4] = 0u;  // counters this block has bumped (bit 0 logits, bit 1 activations)
      s_mask[6] = 0u;
      s_mask[8] = 0u;
    }
    if constexpr (kStack) copy_layer(0);
    __syncthreads();
  }
  // copies of the prologue: bit 0 router rows, bit 1 shared gate/up rows, bit 2
  // shared down rows.  Without PDL h goes first, then the rest in the order they
  // are needed.  With PDL the router rows (needed right after h) go out before
  // the dependency wait, h and then the shared expert's rows (needed once the
  // logits are out) right after it: in a block's copy engine nothing queues
  // ahead of h but the router rows.  (Shared rows before the wait as well put
  // more ahead of h and crowd the previous launch's tail: slower.)
  auto issue = [&](uint32_t which, const DecodeLayer& y) {
    uint32_t issued = 0u;
    if ((which & 1u) && nrr > 0) {
      mbar_expect_tx(&bar[0], (uint32_t)nrr * H * 2);
      uint8_t* rt = G + a.plan.off_rt;
      if (ne > 0) bulk_g2s(rt, y.router + (size_t)e0 * H, (uint32_t)ne * H * 2, &bar[0]);
      if (nrr > ne) bulk_g2s(rt + (size_t)ne * H * 2, y.gate, (uint32_t)H * 2, &bar[0]);
      issued |= 1u;
    }
    if ((which & 2u) && hs && nr > 0) {
      const uint32_t bytes = (uint32_t)nr * s_gu_pair;
      mbar_expect_tx(&bar[1], bytes);
      bulk_g2s(G + a.plan.off_sgu, y.shared + (size_t)r0 * s_gu_pair, bytes, &bar[1]);
      issued |= 2u;
    }
    if ((which & 4u) && hs && nj > 0) {
      const uint32_t bytes = (uint32_t)nj * s_d_row;
      mbar_expect_tx(&bar[1 + NE], bytes);
      bulk_g2s(D, y.shared + s_d_off + (size_t)j0 * s_d_row, bytes, &bar[1 + NE]);
      issued |= 2u << NE;
    }
    return issued;
  };
  auto issue_h = [&]() {
    mbar_expect_tx(&bar[bar_h], (uint32_t)H * 4);
    bulk_g2s(hbuf, a.h, (uint32_t)H * 4, &bar[bar_h]);
    return 1u << bar_h;
  };
  constexpr uint32_t kEarly = 1u;
  if (l == 0) {
    if (tid == 0) s_mask[0] = kPDL ? issue(kEarly, ly()) : (issue_h() | issue(7u, ly()));
    if (kPDL) {
      pdl_launch_dependents();
      pdl_wait_prior();
      if (tid == 0) s_mask[0] |= issue_h() | issue(7u & ~kEarly, ly());
    }
  }

  // one warp waits on mbarrier i (its phase of this layer); a give-up is
  // recorded and acted on at the next block barrier, so that all threads leave
  // together
  auto warp_wait = [&](int i) -> bool {  // none once the block has failed
    const bool ok = *(volatile uint32_t*)&s_mask[1] == 0u && mbar_wait(&bar[i], parity(i));
    if (!ok && lane == 0) atomicOr(&s_mask[1], 1u);
    return __all_sync(0xffffffffu, ok);
  };
  auto failed = [&]() -> bool { return __syncthreads_or(tid == 0 && s_mask[1] != 0u) != 0; };

  // ---- this launch's epoch
  if (l == 0) {
    if (tid == 0) {
      // every block adds one now and, after the last layer, one for every
      // further layer, so this launch's first layer is number count / P
      const unsigned long long n = atomicAdd(&a.hdr->launches, 1ull);
      s_mask[2] = (uint32_t)(n / (unsigned long long)P + 1ull);
      s_mask[3] = *(volatile uint32_t*)&a.hdr->bar_extra;  // test hook: readers expect a later epoch
      // no block of this launch adds to the output-row counter before every
      // block has published its layer-0 activations, which each does after
      // this read (acquire: the read is not reordered after them)
      if constexpr (kStack) *s_hbase = ld_acquire_u64(&a.hdr->published_h);
    }
    if (__syncthreads_or(tid == 0 && *(volatile uint32_t*)&a.hdr->abort)) goto cleanup;
  }
  {
    const uint32_t epoch = s_mask[2] + (uint32_t)l;  // written with every published word
    const uint32_t expect = epoch + s_mask[3];        // awaited by every reader
    float4 hv0, hv1;
    if (!kStack || l == 0) {
      warp_wait(bar_h);
      if (tid == 0) STAMP(1);
      hv0 = 4 * tid < H ? reinterpret_cast<const float4*>(hbuf)[tid] : make_float4(0.f, 0.f, 0.f, 0.f);
      hv1 = 4 * (tid + kBlock) < H ? reinterpret_cast<const float4*>(hbuf)[tid + kBlock] : make_float4(0.f, 0.f, 0.f, 0.f);
      hres = tid < nj ? hbuf[j0 + tid] : 0.f;
      if constexpr (kStack) {
        if (tid < nj) s_hres[tid] = hres;
      }
    } else {
      // ---- input: the previous layer's output rows, published by every
      // block (this block's own rows are already in s_hres).  One
      // thread waits on the counter; every thread then loads its 8 words and
      // polls the late ones together.
      copy_layer(l);
      if (tid == 0) {
        s_mask[8] ^= s_mask[0];  // each barrier the previous layer used has completed one phase
        s_mask[0] = s_mask[6];   // copies for this layer issued during the previous one
        s_mask[6] = 0u;
        s_mask[4] = 0u;
        const bool ok = wait_count(a.hdr, &a.hdr->published_h, *s_hbase + (unsigned long long)P * (l + s_mask[3]));
        s_mask[7] = ok ? 0u : 1u;
      }
      if (__syncthreads_or(tid == 0 && s_mask[7] != 0u)) goto cleanup;
      const uint32_t want = expect - 1u;
      unsigned long long hw[8];
      bool late = false;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int j = 4 * (tid + kBlock * (k >> 2)) + (k & 3);
        hw[k] = j < H ? ld_pub(pub_h + h_slot(j)) : ((unsigned long long)want << 32);  // past H: zero, ready
        late |= !pub_ready(hw[k], want);
      }
      if (late) {
        const unsigned long long t0 = globaltimer();
        int spins = 0;
        while (late) {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (!pub_ready(hw[k], want)) hw[k] = ld_pub(pub_h + h_slot(4 * (tid + kBlock * (k >> 2)) + (k & 3)));
          late = false;
#pragma unroll
          for (int k = 0; k < 8; ++k) late |= !pub_ready(hw[k], want);
          if (late && (++spins & 63) == 0 &&
              (*(volatile uint32_t*)&a.hdr->abort || globaltimer() - t0 > kTimeoutNs)) {
            if (globaltimer() - t0 > kTimeoutNs) {
              atomicOr(&a.hdr->status, ST_TIMEOUT);
              atomicExch(&a.hdr->abort, 1u);
            }
            atomicOr(&s_mask[1], 1u);  // acted on at the block barrier after the router rows
            break;
          }
        }
      }
      hv0 = make_float4(pub_value(hw[0]), pub_value(hw[1]), pub_value(hw[2]), pub_value(hw[3]));
      hv1 = make_float4(pub_value(hw[4]), pub_value(hw[5]), pub_value(hw[6]), pub_value(hw[7]));
    }

    // ---- x = h * gamma and the sum of h^2 (the router needs only these; the
    // limbs of x follow once the logits are out).  Thread t holds values
    // 4t .. 4t+3 and 4(t+512) .. 4(t+512)+3, so warp w holds groups 2w, 2w+1
    // and 2w+16, 2w+17.
    float ss = 0.f;
    {
      float4 xs[2] = {hv0, hv1};
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int i0 = 4 * (tid + kBlock * k);
        float4& x = xs[k];
        ss = fmaf(x.x, x.x, fmaf(x.y, x.y, fmaf(x.z, x.z, fmaf(x.w, x.w, ss))));
        if (ly().gamma && i0 < H) {
          const uint2 gw = *reinterpret_cast<const uint2*>(ly().gamma + i0);
          x.x *= bf16lo(gw.x); x.y *= bf16hi(gw.x); x.z *= bf16lo(gw.y); x.w *= bf16hi(gw.y);
        }
      }
      hv0 = xs[0];
      hv1 = xs[1];
    }
    ss = warp_sum(ss);
    if (lane == 0) s_red[wid] = ss;
    __syncthreads();
    if (tid == 0) STAMP(2);
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) tot += s_red[w];
    const float rs = 1.0f / sqrtf(tot / (float)H + a.eps);  // xn = rs * x

    // ---- gate/up lane geometry; this lane's limbs of x
    const RowMap mh = make_rowmap(ngh);
    const int gchunk = wid % mh.chunks, gnstreams = kWarps / mh.chunks;
    const int gsub = lane % mh.lpr;
    const int gg = gchunk * 32 + gsub;
    const bool ggact = gg < ngh;
    const int gr_warp = (wid / mh.chunks) * mh.rpp;  // first row of the warp (warp-uniform)
    const int gr_first = gr_warp + lane / mh.lpr, gr_step = gnstreams * mh.rpp;
    auto load_x = [&](Limbs& xl, float2& xe) {
      xe = make_float2(0.f, 0.f);
      if (ggact) {
        load_limbs(AL, ngh, gg, xl);
        xe = AE[gg];
      } else {
        zero_limbs(xl);
      }
    };
    // gate/up rows of expert p (slice at `slot`, code width bits) -> partials
    // part[p][r * chunks + chunk]; the warp waits for the slice itself.  The
    // skip test is warp-uniform: the wait and the row reductions are warp
    // collectives, so a warp takes part with all of its lanes or not at all.
    auto gate_up = [&](int p, const uint8_t* slot, auto bits_c, const Limbs& xl, float2 xe) {
      constexpr int kBits = decltype(bits_c)::value;
      if (nr == 0 || gr_warp >= 2 * nr) return;  // no rows for this warp: nothing to wait for
      if (!warp_wait(1 + p)) return;
      float o0, o1;
      if constexpr (kBits == 4)
        slice_rows2<4, true>(slot, f4.gu_row, f4.gu_codes, ngh, gg, ggact, xl, xe, gr_first, gr_step, 2 * nr,
                             mh.lpr, o0, o1);
      else
        slice_rows2<2, true>(slot, f2.gu_row, f2.gu_codes, ngh, gg, ggact, xl, xe, gr_first, gr_step, 2 * nr,
                             mh.lpr, o0, o1);
      if (gsub == 0) {
        float* pb = part + (size_t)p * part_stride;
        if (gr_first < 2 * nr) pb[gr_first * mh.chunks + gchunk] = o0;
        if (gr_first + gr_step < 2 * nr) pb[(gr_first + gr_step) * mh.chunks + gchunk] = o1;
      }
    };

    // ---- router rows -> published logits (each thread's 8 values of x against each row)
    if (nrr > 0) warp_wait(0);
    if (tid == 0) STAMP(3);
    {
      // four rows at a time, their warp reductions interleaved (the same
      // butterfly per row as warp_sum, so the sums do not change)
      const uint8_t* rt = G + a.plan.off_rt;
      for (int rb = 0; rb < nrr; rb += 4) {
        float acc[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int ri = rb + q;
          acc[q] = 0.f;
          if (ri < nrr && 4 * tid < H) {
            const uint2 rw = *reinterpret_cast<const uint2*>(rt + ((size_t)ri * H + 4 * tid) * 2);
            acc[q] = fmaf(bf16lo(rw.x), hv0.x, acc[q]);
            acc[q] = fmaf(bf16hi(rw.x), hv0.y, acc[q]);
            acc[q] = fmaf(bf16lo(rw.y), hv0.z, acc[q]);
            acc[q] = fmaf(bf16hi(rw.y), hv0.w, acc[q]);
          }
          if (ri < nrr && 4 * (tid + kBlock) < H) {
            const uint2 rw = *reinterpret_cast<const uint2*>(rt + ((size_t)ri * H + 4 * (tid + kBlock)) * 2);
            acc[q] = fmaf(bf16lo(rw.x), hv1.x, acc[q]);
            acc[q] = fmaf(bf16hi(rw.x), hv1.y, acc[q]);
            acc[q] = fmaf(bf16lo(rw.y), hv1.z, acc[q]);
            acc[q] = fmaf(bf16hi(rw.y), hv1.w, acc[q]);
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], o);
        if (lane == 0) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (rb + q < nrr) rpart[(rb + q) * kWarps + wid] = acc[q];
        }
      }
    }
    if (failed()) goto cleanup;
    if (wid == 0) {
      if (lane < nrr) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) v += rpart[lane * kWarps + w];
        v *= rs;
        const int e = lane < ne ? e0 + lane : E;  // the shared-gate logit is row E
        if (e < E && ly().offset) v += ly().offset[e];
        st_pub(a.pub_logits + e, v, epoch);
      }
      __syncwarp();
      if (lane == 0) {
        red_relaxed_add_u64(&a.hdr->published_logits, 1ull);
        STAMP(4);
        s_mask[4] |= 1u;
      }
    }
    // ---- limbs of x (both passes quantised together), first needed by the
    // gate/up rows: after the logits are out, off the way to top-K
    bool finite = true;
    {
      float4 xs[2] = {hv0, hv1};
      bool st[2];
      int gs[2];
      uint8_t* vs[2] = {AL, AL};
      float2* es[2];
      const float one[2] = {1.0f, 1.0f};
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int i0 = 4 * (tid + kBlock * k);
        st[k] = i0 < H;
        gs[k] = st[k] ? i0 / kGroup : 0;
        es[k] = AE + gs[k];
      }
      if (4 * 32 * wid < H)  // the warp's first pass has values (whole warps skip)
        finite = quantize_groups<2>(xs, lane, st, vs, ngh, gs, es, one);
    }
    const int nonfinite_x = __syncthreads_or(!finite);

    // routed gate/up copies of experts k0 .. k1 - 1 (lane 0 of warp 0)
    auto issue_routed = [&](int k0, int k1) {
      uint32_t issued = s_mask[0];
      for (int k = k0; k < k1; ++k) {
        const uint8_t* blob = ly().experts + (size_t)s_idx[k] * ly().stride;
        if (nr > 0) {
          const uint32_t bytes = (uint32_t)nr * r_gu_pair;
          mbar_expect_tx(&bar[1 + hs + k], bytes);
          bulk_g2s(G + (size_t)k * gu_slot, blob + (size_t)r0 * r_gu_pair, bytes, &bar[1 + hs + k]);
          issued |= 2u << (hs + k);
        }
      }
      s_mask[0] = issued;
    };
    // ---- shared expert gate/up (its rows were staged first): warps 1.. now,
    // warp 0 once it has routed the token (below)
    auto shared_gate_up = [&]() {
      if (hs) {
        Limbs xl;
        float2 xe;
        load_x(xl, xe);
        gate_up(0, G + a.plan.off_sgu, std::integral_constant<int, kSB>{}, xl, xe);
      }
    };
    // Routed gate/up slice k goes to slot k of the gate/up area.  Slots that do
    // not overlap the shared slice (the router rows and h there are dead once
    // the logits are out) are copied right after top-K; slots 0 .. k_late - 1,
    // which the shared slice covers, once every warp is done with it.
    const size_t shared_end = hs ? a.plan.off_sgu + (size_t)nr * s_gu_pair : 0;
    const int k_late = min(K, (int)((shared_end + gu_slot - 1) / gu_slot));
    {
      // ---- routing, by warp 0 of every block (same logits, same result),
      // while the other warps compute the shared rows; they then arrive on
      // named barrier 1 without waiting and go on to the routed rows.
      if (wid != 0) {
        shared_gate_up();
        named_arrive(1, kBlock);
      }
      if (wid == 0) {
        if (lane == 0) STAMP(5);
        bool ok = true;
        bool ready = true;  // the words carry their epoch: polled directly
        if (lane == 0) STAMP(6);
        ready = __all_sync(0xffffffffu, ready);
        uint32_t key[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) key[i] = 0u;
        // logits of this launch: lane l reads experts l, l + 32, ... (all of
        // its words in flight together; a word not yet visible is polled again)
        const int mine = E > lane ? (E - lane + 31) / 32 : 0;
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          if (ch * 16 < mine && ready) {  // lane-dependent, no collectives inside
            float v[16];
            ready = poll_pub<16>(a.hdr, a.pub_logits + lane + 512 * ch, 32, min(16, mine - ch * 16), expect, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              if (ch * 16 + i < mine) {
                ok &= isfinite(v[i]);
                key[ch * 16 + i] = fkey(v[i]);
              }
            }
          }
        }
        float gate_logit = 0.f;
        if (lane == 0 && a.has_gate && ready) {
          float v[1];
          ready = poll_pub<1>(a.hdr, a.pub_logits + E, 1, 1, expect, v);
          gate_logit = v[0];
        }
        if (__all_sync(0xffffffffu, ready)) {
          if (E <= 128) {
            uint32_t k4[4] = {key[0], key[1], key[2], key[3]};
            warp_topk<4>(k4, K, lane, s_idx, s_val);
          } else if (E <= 512) {
            uint32_t k16[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) k16[i] = key[i];
            warp_topk<16>(k16, K, lane, s_idx, s_val);
          } else {
            warp_topk<32>(key, K, lane, s_idx, s_val);
          }
          ok = __all_sync(0xffffffffu, ok);
          if (lane == 0) {
            // the generic-proxy reads of the router rows and h are complete
            // (block barrier after the router rows)
            fence_proxy_async();
            issue_routed(k_late, K);
            STAMP(7);
            chosen_softmax(s_val, K, s_coef + hs);
            if (hs) s_coef[0] = a.has_gate ? 1.0f / (1.0f + expf(-gate_logit)) : 1.0f;
            if (c == 0) {
              if (!ok || nonfinite_x) atomicOr(&a.hdr->status, ST_NONFINITE);
              for (int k = 0; k < K; ++k) {
                if (ly().idx_out) ly().idx_out[k] = s_idx[k];
                if (ly().w_out) ly().w_out[k] = s_coef[hs + k];
              }
            }
          }
        } else if (lane == 0) {
          atomicOr(&s_mask[1], 1u);
        }
        __syncwarp();
        // this warp's shared rows, then the copies over the shared slice once
        // every warp is done with it (only if routing succeeded: s_idx is
        // written by top-K)
        shared_gate_up();
        named_sync(1, kBlock);
        if (lane == 0 && k_late > 0 && *(volatile uint32_t*)&s_mask[1] == 0u) {
          fence_proxy_async();  // the generic-proxy reads of the shared rows are complete
          issue_routed(0, k_late);
        }
        __syncwarp();
      }
    }
    {
      // ---- routed gate/up rows, in the order the copies were issued
      Limbs xl;
      float2 xe;
      load_x(xl, xe);
      for (int i = 0; i < K; ++i) {
        const int k = (i + k_late) % K;  // early slots first, as their copies went out
        gate_up(hs + k, G + (size_t)k * gu_slot, std::integral_constant<int, kRB>{}, xl, xe);
        if (tid == 0) STAMP(8 + i);
        // routed down rows are needed last: warp 0 issues expert k's copy once
        // its gate/up rows have landed (warp 0 has gate/up rows whenever the
        // block has any, and gate_up waited for them), which keeps the copies
        // in flight per SM few
        // (only if routing succeeded: s_idx is written by top-K; this thread
        // raised the failure flag itself when it did not)
        if (wid == 0 && lane == 0 && nj > 0 && *(volatile uint32_t*)&s_mask[1] == 0u) {
          const uint8_t* blob = ly().experts + (size_t)s_idx[k] * ly().stride;
          const uint32_t bytes = (uint32_t)nj * r_d_row;
          mbar_expect_tx(&bar[1 + NE + hs + k], bytes);
          bulk_g2s(D + (size_t)(hs + k) * dn_slot, blob + r_d_off + (size_t)j0 * r_d_row, bytes, &bar[1 + NE + hs + k]);
          s_mask[0] |= 2u << (NE + hs + k);
        }
      }
    }

    // ---- SwiGLU of every expert's rows, weighted by the expert's routing
    // coefficient, published for every block
    if (failed()) goto cleanup;
    if (tid == 0) STAMP(16);
    if constexpr (kStack) {
      // the routed gate/up slices are dead: the next layer's router rows and
      // shared gate/up rows go to the gate/up area now (the down partials lie
      // past both)
      if (tid == kPrefetchTid && l + 1 < nlayers) {
        fence_proxy_async();  // the generic-proxy reads of the slices are complete (block barrier)
        s_mask[6] = issue(3u, s_ly[1]);
      }
    }
    for (int t = tid; t < NE * nr; t += kBlock) {
      const int p = t / nr, i = t - p * nr;
      const float* pb = part + (size_t)p * part_stride;
      float gsum = 0.f, usum = 0.f;
      for (int ch = 0; ch < mh.chunks; ++ch) {
        gsum += pb[(2 * i) * mh.chunks + ch];
        usum += pb[(2 * i + 1) * mh.chunks + ch];
      }
      st_pub(a.pub_act + (size_t)p * I + act_slot(r0 + i), s_coef[p] * silu_mul(rs * gsum, rs * usum), epoch);
    }
    __syncthreads();
    if (tid == 0) {
      red_relaxed_add_u64(&a.hdr->published_act, 1ull);
      s_mask[4] |= 2u;
    }
    // activation reader: one thread waits on the counter, then every thread
    // loads the words it needs and polls the late ones again.  (Polling the
    // words without the counter, as for the logits, cost 3.7 us a token on
    // B300: 148 blocks re-reading 40 KB each while others still compute.)
    if (tid == 0) {
      STAMP(17);
      const bool ok = wait_count(a.hdr, &a.hdr->published_act, (unsigned long long)P * expect);
      STAMP(18);
      s_mask[5] = ok ? 0u : 1u;
    }
    if (__syncthreads_or(tid == 0 && s_mask[5] != 0u)) goto cleanup;
    if (tid == 0) STAMP(19);

    // ---- limbs of every weighted a: a half-warp per group, 2 groups per warp
    // per pass, kActPasses passes quantised together
    {
      constexpr int kActPasses = 3;
      bool fin = true, ready = true;
      const int ngroups = NE * ngi;
      for (int base0 = 2 * wid; base0 < ngroups; base0 += 2 * kWarps * kActPasses) {
        float4 xs[kActPasses];
        bool st[kActPasses];
        int gs[kActPasses];
        uint8_t* vs[kActPasses];
        float2* es[kActPasses];
        float one[kActPasses];
        size_t w0s[kActPasses];
        unsigned long long wv[kActPasses][4];
        bool late = false;
#pragma unroll
        for (int k = 0; k < kActPasses; ++k) {
          const int gi = base0 + 2 * kWarps * k + (lane >> 4);
          st[k] = gi < ngroups;
          const int gq = st[k] ? gi : 0;  // an idle half takes part in the shuffles
          const int p = gq / ngi, g = gq - p * ngi;
          gs[k] = g;
          vs[k] = AL + (size_t)p * ngi * kLimbBytes;
          es[k] = AE + (size_t)p * ngi + g;
          one[k] = 1.0f;
          // values 4j .. 4j+3 of the group sit at slots j, j + 16, j + 32, j + 48
          w0s[k] = (size_t)p * I + g * kGroup + (lane & 15);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            wv[k][i] = ld_pub(a.pub_act + w0s[k] + 16 * i);
            late |= !pub_ready(wv[k][i], expect);
          }
        }
        // words that were not yet visible when the copy ran: polled again, all
        // of this thread's together
        if (late && ready) {
          const unsigned long long t0 = globaltimer();
          int spins = 0;
          while (late) {
            late = false;
#pragma unroll
            for (int k = 0; k < kActPasses; ++k)
#pragma unroll
              for (int i = 0; i < 4; ++i)
                if (!pub_ready(wv[k][i], expect)) wv[k][i] = ld_pub(a.pub_act + w0s[k] + 16 * i);
#pragma unroll
            for (int k = 0; k < kActPasses; ++k)
#pragma unroll
              for (int i = 0; i < 4; ++i) late |= !pub_ready(wv[k][i], expect);
            if (late && (++spins & 63) == 0) {
              if (*(volatile uint32_t*)&a.hdr->abort || globaltimer() - t0 > kTimeoutNs) {
                if (globaltimer() - t0 > kTimeoutNs) {
                  atomicOr(&a.hdr->status, ST_TIMEOUT);
                  atomicExch(&a.hdr->abort, 1u);
                }
                ready = false;
                break;
              }
            }
          }
        }
#pragma unroll
        for (int k = 0; k < kActPasses; ++k)
          xs[k] = make_float4(pub_value(wv[k][0]), pub_value(wv[k][1]), pub_value(wv[k][2]), pub_value(wv[k][3]));
        fin &= quantize_groups<kActPasses>(xs, lane, st, vs, ngi, gs, es, one);
      }
      if (!ready) atomicOr(&s_mask[1], 1u);
      if (__syncthreads_or(!fin) && tid == 0) atomicOr(&a.hdr->status, ST_NONFINITE);
    }
    if (failed()) goto cleanup;
    if (tid == 0) STAMP(20);

    // ---- down rows of every expert as one long dot product per row: thread
    // (set, q) takes unit q = (expert p, group g) of rows set, set + S, ...;
    // partials go to pdn[row][q] and are summed in a fixed order
    {
      const int Q = NE * ngi, S = kBlock / Q;
      const int set = tid / Q, q = tid - set * Q;
      if (set < S && set < nj) {
        const int p = q / ngi, g = q - p * ngi;
        // lanes of one warp may belong to different experts: each thread waits
        // for its own expert's rows (no warp collective in this section)
        if (!mbar_wait(&bar[1 + NE + p], parity(1 + NE + p))) atomicOr(&s_mask[1], 1u);
        Limbs L;
        load_limbs(AL + (size_t)p * ngi * kLimbBytes, ngi, g, L);
        const float2 es = AE[(size_t)p * ngi + g];
        const uint8_t* base = D + (size_t)p * dn_slot;
        // up to kDnRows independent rows per thread, interleaved for ILP
        auto rows = [&](auto bits_c) {
          constexpr int kBits = decltype(bits_c)::value;
          const Fmt& f = kBits == 4 ? f4 : f2;
#pragma unroll
          for (int k = 0; k < kDnRows; ++k) {
            const int r = set + k * S;
            if (r < nj) pdn[r * Q + q] = row_group<kBits>(base + (size_t)r * f.d_row, ngi, f.d_codes, g, L, es);
          }
        };
        if constexpr (kSB == kRB)
          rows(std::integral_constant<int, kRB>{});
        else if (p < hs)
          rows(std::integral_constant<int, kSB>{});
        else
          rows(std::integral_constant<int, kRB>{});
      }
      if (failed()) goto cleanup;
      if (tid == 0) STAMP(21);
      if constexpr (kStack) {
        // the down slices are dead: the next layer's shared down rows go to slot 0
        if (tid == kPrefetchTid && l + 1 < nlayers) {
          fence_proxy_async();
          s_mask[6] |= issue(4u, s_ly[1]);
        }
      }
      // row r: 16 threads sum every 16th partial, then a butterfly over the 16
      {
        const int r = tid >> 4, sub = tid & 15;
        float v = 0.f;
        if (r < nj)
          for (int qq = sub; qq < Q; qq += 16) v += pdn[r * Q + qq];
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (sub == 0 && r < nj) ysm[r] = v;
      }
      __syncthreads();
      // ---- output rows (warp 0's lanes: nj <= 32): h += y after the last
      // layer, else published as the next layer's input
      if (wid == 0) {
        if (lane < nj) {
          const float hn = (kStack ? s_hres[lane] : hres) + ysm[lane];
          if (l + 1 == nlayers)
            a.h[j0 + lane] = hn;
          else
            st_pub(pub_h + h_slot(j0 + lane), hn, epoch);
          if constexpr (kStack) s_hres[lane] = hn;
        }
        if (kStack && l + 1 < nlayers) {
          __syncwarp();
          if (lane == 0) red_relaxed_add_u64(&a.hdr->published_h, 1ull);
        }
      }
      if (tid == 0) STAMP(22);
    }
  }
  if constexpr (kStack) {
    // the launch's further layers, counted once its last layer is done
    if (tid == 0 && l + 1 == nlayers && nlayers > 1)
      red_relaxed_add_u64(&a.hdr->launches, (unsigned long long)(nlayers - 1));
  }
  return true;

cleanup:
  // leave only after this block's own copies in flight have landed, and with
  // the epoch counters advanced by this block as in a complete launch (one per
  // layer: those of the layer that failed still owed, and all of the later
  // layers').  The output-row counter needs nothing: a stack launch reads it
  // afresh.
  __syncthreads();
  if (tid == 0) {
    const unsigned long long later = (unsigned long long)(nlayers - 1 - l);
    const uint32_t bumped = s_mask[4];
    const unsigned long long owed_lg = (bumped & 1u ? 0ull : 1ull) + later;
    const unsigned long long owed_act = (bumped & 2u ? 0ull : 1ull) + later;
    if (owed_lg) red_relaxed_add_u64(&a.hdr->published_logits, owed_lg);
    if (owed_act) red_relaxed_add_u64(&a.hdr->published_act, owed_act);
    if (nlayers > 1) red_relaxed_add_u64(&a.hdr->launches, (unsigned long long)(nlayers - 1));
    // copies of this layer, and (stack) those already issued for the next one,
    // which complete the following phase of their barrier
    const uint32_t issued = s_mask[0], next = s_mask[6], ph = kStack ? s_mask[8] : 0u;
    for (int i = 0; i < nbar; ++i) {
      if (issued >> i & 1u) mbar_wait(&bar[i], (ph >> i) & 1u);
      if (next >> i & 1u) mbar_wait(&bar[i], ((ph ^ issued) >> i) & 1u);
    }
  }
  __syncthreads();
  return false;
}

template <bool kPDL, int kRB, int kSB>
__global__ void __launch_bounds__(kBlock, 1) decode_b1_kernel(const __grid_constant__ DecodeArgs a) {
  decode_body<kPDL, kRB, kSB, false>(a, nullptr, 1, nullptr, 0);
}

template <bool kPDL, int kRB, int kSB>
__global__ void __launch_bounds__(kBlock, 1) decode_stack_kernel(const __grid_constant__ StackArgs a) {
  // one body for every layer: its code stays in the instruction cache (a copy
  // of the body specialised for layer 0 cost ~40 us a launch in instruction
  // fetches)
  for (int l = 0; l < a.L; ++l)
    if (!decode_body<kPDL, kRB, kSB, true>(a.d, a.layers, a.L, a.pub_h, l)) return;
}

#ifdef MOE_TIMELINE
extern "C" int moe_timeline_read(unsigned long long* host, int n) {
  return (int)cudaMemcpyFromSymbol(host, g_timeline, sizeof(unsigned long long) * (size_t)n);
}
#endif

bool decode_plan_for(int nsm, int optin, int H, int I, int E, int K, int bits, int shared_bits, int has_shared,
                     int has_gate, DecodePlan* out) {
  const int NE = K + has_shared;
  if (H > 4096 || I > 2048 || E > 1024 || K > kMaxTopK || nsm < 1) return false;
  const Fmt fr = make_fmt(bits, H, I);
  const Fmt fs = make_fmt(has_shared ? shared_bits : bits, H, I);
  const RowMap mh = make_rowmap(fr.ng_h), mi = make_rowmap(fr.ng_i);
  if (kWarps % mh.chunks || mi.chunks != 1) return false;
  DecodePlan p{};
  p.P = nsm;
  p.rows_gu = (I + nsm - 1) / nsm;
  p.rows_d = (H + nsm - 1) / nsm;
  p.rows_r = (E + nsm - 1) / nsm + (has_gate ? 1 : 0);
  // each warp covers at most two gate/up rows and two down rows per expert;
  // SwiGLU rows and router rows are finished by one warp
  if (2 * p.rows_gu > 2 * (kWarps / mh.chunks) * mh.rpp) return false;
  if (p.rows_d > 2 * kWarps * mi.rpp) return false;
  if (p.rows_gu > 32 || p.rows_r > 32 || p.rows_d > kBlock / 16) return false;
  {
    const int Q = NE * fr.ng_i, S = Q > 0 ? kBlock / Q : 0;
    if (S < 1 || p.rows_d > kDnRows * S) return false;
  }
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = (o + bytes + 127) & ~size_t(127);
    return at;
  };
  // down slices, one slot per expert (slot 0 the shared expert when present)
  p.dn_slot = pad16((size_t)p.rows_d * std::max(fr.d_row, fs.d_row));
  p.off_dn = take((size_t)NE * p.dn_slot);
  // gate/up area: the K routed slices, or (before routing) the shared slice
  // and the router rows (offsets relative to the area)
  p.gu_slot = pad16((size_t)p.rows_gu * fr.gu_pair);
  size_t pre = 0;
  auto sub = [&](size_t bytes) {
    const size_t at = pre;
    pre = (pre + bytes + 127) & ~size_t(127);
    return at;
  };
  p.off_sgu = sub(has_shared ? (size_t)p.rows_gu * fs.gu_pair : 0);
  p.off_rt = sub((size_t)p.rows_r * H * 2);
  p.off_hbuf = sub((size_t)H * 4);  // h, one bulk copy (first layer)
  // after the gate/up phase: the down partials, past the shared slice and the
  // router rows (where a stack launch copies the next layer's while the down
  // partials are in use); h is dead by then
  p.off_pdn = p.off_hbuf;
  const size_t post = ((size_t)p.rows_d * NE * fr.ng_i * 4 + 127) / 128 * 128;
  p.off_g = take(std::max(std::max(pre, (size_t)K * p.gu_slot), p.off_pdn + post));
  // limbs: of x first (read into registers), later of every expert's activation
  const size_t ngroups = std::max((size_t)NE * fr.ng_i, (size_t)fr.ng_h);
  p.off_al = take(ngroups * kLimbBytes);
  p.off_ae = take(ngroups * 8);
  p.part_stride = 2 * p.rows_gu * mh.chunks;
  p.off_part = take((size_t)NE * p.part_stride * 4);
  p.off_rpart = take((size_t)p.rows_r * kWarps * 4);
  p.off_y = take((size_t)p.rows_d * 4);
  p.off_bar = take((size_t)(1 + 2 * NE + 1) * 8);
  // scalars, then (stack) the layer's pointers and the block's input rows
  p.off_misc = take(256 + 2 * sizeof(DecodeLayer) + 32 * 4);
  p.total = o + 128;  // slack for rounding the dynamic base up to 128 bytes
  if (p.total > (size_t)optin) return false;
  *out = p;
  return true;
}

bool decode_plan(int H, int I, int E, int K, int bits, int shared_bits, int has_shared, int has_gate, int device,
                 DecodePlan* out) {
  int nsm = 0, optin = 0;
  if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess) return false;
  return decode_plan_for(nsm, optin, H, I, E, K, bits, shared_bits, has_shared, has_gate, out);
}

namespace {
// the instantiation for (PDL, routed bits, shared bits); without a shared
// expert the shared width is the routed one
template <bool kPDL, bool kStack>
auto decode_kernel_for(int bits, int shared_bits) {
  if constexpr (kStack) {
    if (bits == 4) return shared_bits == 4 ? decode_stack_kernel<kPDL, 4, 4> : decode_stack_kernel<kPDL, 4, 2>;
    return shared_bits == 4 ? decode_stack_kernel<kPDL, 2, 4> : decode_stack_kernel<kPDL, 2, 2>;
  } else {
    if (bits == 4) return shared_bits == 4 ? decode_b1_kernel<kPDL, 4, 4> : decode_b1_kernel<kPDL, 4, 2>;
    return shared_bits == 4 ? decode_b1_kernel<kPDL, 2, 4> : decode_b1_kernel<kPDL, 2, 2>;
  }
}

template <bool kStack, class Args>
cudaError_t launch_any(const Args& args, const DecodeArgs& a, bool pdl, cudaStream_t s) {
  static std::atomic<int> configured[2][4][kMaxDevices];  // per PDL variant, code widths and device
  const int bytes = (int)a.plan.total;
  const int sb = a.has_shared ? a.shared_bits : a.bits;
  const int v = (a.bits == 4 ? 0 : 2) + (sb == 4 ? 0 : 1);
  const auto kp = decode_kernel_for<true, kStack>(a.bits, sb);
  const auto kn = decode_kernel_for<false, kStack>(a.bits, sb);
  const cudaError_t e = pdl ? ensure_dynamic_smem(kp, bytes, configured[1][v])
                            : ensure_dynamic_smem(kn, bytes, configured[0][v]);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.plan.P);
  cfg.blockDim = dim3(kBlock);
  cfg.dynamicSmemBytes = (size_t)bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    // one block per SM (shared memory forces it) and one wave: every block is
    // resident once the previous kernel's blocks have left
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  } else {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return pdl ? cudaLaunchKernelEx(&cfg, kp, args) : cudaLaunchKernelEx(&cfg, kn, args);
}
}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, bool pdl, cudaStream_t s) { return launch_any<false>(a, a, pdl, s); }

cudaError_t launch_decode_stack(const StackArgs& a, bool pdl, cudaStream_t s) {
  if (a.L < 1 || a.L > kMaxStackLayers) return cudaErrorInvalidValue;
  return launch_any<true>(a, a.d, pdl, s);
}

}  // namespace moe
