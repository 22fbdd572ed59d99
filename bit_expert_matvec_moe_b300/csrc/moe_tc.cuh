// Tensor-core building blocks of the batched expert contraction (sm_103a):
// tcgen05 (MMA into tensor memory), TMA tensor copies and the operand
// descriptors, plus the layout helpers the kernels and the host checks share.
//
// Arithmetic of the batched contraction
// -------------------------------------
// For one expert and a block of up to kTcTok tokens the kernels evaluate
// D[r][t] = sum_c W[r][c] * x_t[c] on the fifth-generation tensor cores
// (kind::f16, fp32 accumulation in tensor memory):
//   * A (M = 128 weight rows x K) holds the dequantised weights
//     W = q * s + b, rounded once to fp16.  The codes are small integers and
//     s, b are bf16 (8 significant bits), so q*s + b needs at most ~13
//     significant bits: the fp16 rounding (11 bits) is nearly exact.  This is
//     the affine dequantisation "nibble * scale + bias" of the page "397B MoE
//     sur MacBook : 4,4 t/s Moteur Flash-MoE" ("Techniques de rupture" item 2),
//     done per weight because the tensor core needs the weights themselves.
//   * B (N = 2 * tokens rows x K) holds each token's activation as two fp16
//     rows, hi = fp16(x') and lo = fp16(x' - hi), x' = x * 2^-e with one power
//     of two per token so that max |x'| lies in [2^14, 2^15): hi + lo carries
//     22 significant bits of every element.  Column 2t of D is the hi part of
//     token t, column 2t + 1 its lo part; the epilogue adds the two and
//     multiplies by 2^e.
// The only roundings are the fp16 weight (relative 2^-11 at most, often 0)
// and the fp32 accumulation.  The tensor core's own fp32 accumulation loses
// low bits at every MMA step (measured on B300: summed over all 4096 inputs of
// a gate/up row in one accumulator, the expert output errs by ~2e-3 by the
// tests' relative-error measure, the bar itself).  So each accumulator spans
// only kSpanKB K-blocks (512 inputs); the epilogue adds the partial sums in
// fp32 registers.  Measured on B300 over 64 skewed-routing tokens of the
// full-width layer (max relative error of y / of y - h): spans of 256 inputs
// 4.7e-4 / 2.7e-4, 512 inputs 4.9e-4 / 6.6e-4, 1024 inputs 9.9e-4 / 1.1e-3;
// each doubling saves 8 % / 2 % of the batch-128 layer call (fewer span
// boundaries in the MMA loop), so 512 keeps a 3x margin under the bar.  bf16
// weights (8 bits) would not meet 2e-3 even with exact sums.
//
// Operand layouts (shared memory, K-major, 128-byte swizzle)
// ----------------------------------------------------------
// A K-block is 64 inputs = one quantisation group.  Each operand row of a
// K-block is 128 bytes (64 fp16), rows in atoms of 8 (1024 bytes); the
// 16-byte chunk c of row r is stored at chunk position c ^ (r & 7) - the
// layout the TMA engine writes with CU_TENSOR_MAP_SWIZZLE_128B and the one
// the MMA reads through a descriptor with swizzle mode "128B".
// Inside each 8-input chunk the inputs are stored in the order
// chunk_perm = {0, 4, 1, 5, 2, 6, 3, 7}: that is the order in which one 32-bit
// code word unpacks into four fp16 pairs (byte j of a 4-bit word holds inputs
// 2j and 2j+1, so masking bytes 0/2 and 1/3 gives the pairs (0,4), (1,5),
// (2,6), (3,7)); the activation rows are written in the same order, so the
// contraction is unchanged.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace moe {
struct WsHeader;
namespace tc {

// status bits of this path (beside ST_TIMEOUT / ST_NONFINITE)
constexpr uint32_t ST_RANGE = 4u;  // a dequantised weight outside the fp16 range
constexpr uint32_t ST_PLAN = 8u;   // more chunks than the work list holds
constexpr uint32_t ST_BOUNDS = 16u;  // an entry or (token, slot) id outside its buffer (access skipped)

constexpr int kTcM = 128;            // weight rows per tile (MMA M)
constexpr int kTcTok = 32;           // tokens per unit at most (MMA N = 2 * tokens <= 64)
constexpr int kStageGroups = 8;      // groups per code stage (one TMA box = 128 bytes of codes per row)
constexpr int kCodeSlots = 3;        // code stages in flight
constexpr int kKSlots = 8;           // K-blocks in flight (A in tensor memory, B in shared memory)
constexpr int kSpanKB = 8;           // K-blocks summed in one accumulator before the epilogue takes it
constexpr int kDBufs = 4;            // accumulators in tensor memory (a ring of partial sums)
constexpr int kDCols = 64;           // tensor-memory columns per accumulator (N <= 64)
constexpr int kTmemACol0 = kDBufs * kDCols;  // A operand: one 32-column block (64 fp16 per lane) per K slot
constexpr int kTmemCols = 512;               // allocation (power of two >= 32)
static_assert(kTmemACol0 + kKSlots * 32 <= kTmemCols, "tensor-memory plan");

constexpr uint32_t kABytes = kTcM * 128;               // 16 KB: one K-block of A (in tensor memory: 32 columns)
constexpr uint32_t kBBytes = 2 * kTcTok * 128;          // 8 KB: one K-block of B at N = 64
constexpr uint32_t kKSlotBytes = kBBytes;              // 8 KB: B only (A lives in tensor memory)
constexpr uint32_t kHalfBoxBytes = kTcM * 128;          // 16 KB: 8 groups' 16-byte code pieces x 128 rows
constexpr uint32_t kSbBoxBytes = kTcM * 32;             // 4 KB: 8 groups' (scale, bias) words x 128 rows
constexpr uint32_t kCodeSlotBytes = 2 * kHalfBoxBytes + kSbBoxBytes;  // 36 KB
constexpr uint32_t kBBoxRows = 16;                      // TMA box of B: 8 tokens x (hi, lo)
constexpr uint32_t kBBoxBytes = kBBoxRows * 128;

// warp roles of the contraction kernel
constexpr int kWarpCodes = 0;     // TMA producer of the code / (scale, bias) stages
constexpr int kWarpB = 1;         // TMA producer of the activation K-blocks
constexpr int kWarpMma = 2;       // tensor-memory owner and MMA issuer
constexpr int kWarpEpi0 = 3;      // 4 epilogue warps (one per tensor-memory lane quarter)
constexpr int kWarpDeq0 = 7;      // 8 dequantising warps
constexpr int kTcWarps = 15;
constexpr int kTcThreads = kTcWarps * 32;

// shared-memory plan (offsets from a 1024-byte aligned base)
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffCodes = kOffK + kKSlots * kKSlotBytes;
constexpr uint32_t kOffBars = kOffCodes + kCodeSlots * kCodeSlotBytes;
constexpr int kNumBars = 2 * kCodeSlots + 2 * kKSlots + 2 * kDBufs + 1;
constexpr uint32_t kOffMisc = kOffBars + 8 * kNumBars;
constexpr uint32_t kSmemUsed = kOffMisc + 64;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // slack for aligning the base
static_assert(kKSlotBytes % 1024 == 0 && kCodeSlotBytes % 1024 == 0, "swizzled regions need 1024-byte alignment");
static_assert(kSmemBytes <= 232448, "contraction kernel exceeds the opt-in shared memory");

__host__ __device__ constexpr int chunk_perm(int p) { return (p >> 1) + 4 * (p & 1); }

// byte offset of 16-byte chunk c of row r inside a 128-byte-swizzled tile
__host__ __device__ constexpr uint32_t swz128(uint32_t r, uint32_t c) {
  return r * 128u + (((c ^ (r & 7u)) & 7u) << 4);
}

// Instruction descriptor of tcgen05.mma kind::f16: fp16 A and B, both
// K-major, fp32 accumulator, M x N (M = 64/128, N multiple of 16 for M = 128).
// Fields (PTX ISA, "Instruction descriptor" of tcgen05.mma): [4,6) D format
// (1 = f32), [7,10) A format (0 = f16), [10,13) B format (0 = f16), bit 15 / 16
// A / B major (0 = K), [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t make_idesc_f16(int M, int N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (0u << 15) | (0u << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor (tcgen05 form): [0,14) start address >> 4,
// [16,30) leading byte offset >> 4, [32,46) stride byte offset >> 4,
// [46,48) version = 1, [49,52) base offset, bit 52 LBO mode, [61,64) swizzle
// (2 = 128-byte).  For a K-major 128-byte-swizzled operand the stride byte
// offset is the distance between 8-row atoms (1024) and the leading byte
// offset is not used (1 by convention).
constexpr uint32_t kSwizzle128 = 2;
__host__ __device__ constexpr uint64_t make_sdesc(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                                  uint32_t swizzle) {
  return (uint64_t)((smem_addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)(swizzle & 7u) << 61);
}
__host__ __device__ constexpr uint64_t sdesc_sw128_kmajor(uint32_t smem_addr) {
  return make_sdesc(smem_addr, 16, 1024, kSwizzle128);
}

// Unpacking one 32-bit code word into fp16 pairs.  Field spec f selects
// (word >> shift) & mask; each 16-bit half then holds m * q for one input
// (m = the field's position weight), OR-ed into the mantissa of 1024.0
// (0x6400) it reads as the fp16 value 1024 + m*q exactly, and
// fma(that, inv_m, neg_off) with inv_m = 1/m, neg_off = -1024/m gives q exactly.
// Pair f of a 4-bit word holds inputs (f, f + 4) of the word's 8 inputs; pair f
// of a 2-bit word (16 inputs) holds inputs (f, f + 4) for f < 4 and
// (f + 4, f + 8) for f >= 4 - always the order chunk_perm within each chunk.
struct FieldSpec {
  uint32_t shift, mask, inv_m, neg_off;
};
constexpr uint32_t kMagic1024 = 0x64006400u;
constexpr uint32_t kOne = 0x3C003C00u, kM1024 = 0xE400E400u;  // 1, -1024
constexpr uint32_t kInv4 = 0x34003400u, kM256 = 0xDC00DC00u;  // 1/4, -256
constexpr uint32_t kInv16 = 0x2C002C00u, kM64 = 0xD400D400u;  // 1/16, -64
constexpr uint32_t kInv64 = 0x24002400u, kM16 = 0xCC00CC00u;  // 1/64, -16
constexpr FieldSpec kField4[4] = {
    {0, 0x000F000Fu, kOne, kM1024}, {0, 0x00F000F0u, kInv16, kM64}, {8, 0x000F000Fu, kOne, kM1024},
    {8, 0x00F000F0u, kInv16, kM64}};
constexpr FieldSpec kField2[8] = {
    {0, 0x00030003u, kOne, kM1024}, {0, 0x000C000Cu, kInv4, kM256}, {8, 0x00030003u, kOne, kM1024},
    {8, 0x000C000Cu, kInv4, kM256}, {0, 0x00300030u, kInv16, kM64}, {0, 0x00C000C0u, kInv64, kM16},
    {8, 0x00300030u, kInv16, kM64}, {8, 0x00C000C0u, kInv64, kM16}};

// Code pieces of stage st (groups 8st .. 8st+7) inside a row's code bytes:
// byte offsets of the first-half and second-half 16-byte pieces of group 8st
// (4-bit; the eight groups' pieces are contiguous, 128 bytes) or of the
// group's whole 16 bytes (2-bit, x1 unused).  Mirrors the packed layout:
// chunks of up to 32 groups, first halves of the chunk, then second halves.
__host__ __device__ inline void stage_code_x(int bits, int ng, int st, int* x0, int* x1) {
  const int g = kStageGroups * st;
  if (bits == 4) {
    const int k = g >> 5, i = g & 31;
    const int n = (ng - 32 * k) < 32 ? (ng - 32 * k) : 32;
    *x0 = 1024 * k + 16 * i;
    *x1 = 1024 * k + 16 * (n + i);
  } else {
    *x0 = 16 * g;
    *x1 = 16 * g;
  }
}

// Units of work: (chunk of at most kTcTok entries of one expert, 128-row tile).
struct TcChunk {
  int expert;  // routed expert id, or -1 for the shared expert
  int e0;      // first entry (position in the bucketed entry list)
  int n;       // entries (tokens) in the chunk, 1 .. kTcTok
  int bits;    // code width of the expert
};


// ---------------------------------------------------------------------------
// device wrappers (inline PTX)
// ---------------------------------------------------------------------------
#if defined(__CUDACC__)
__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// TMA tensor copies, global -> shared, completion counted on an mbarrier
__device__ __forceinline__ void tma_load_2d(void* dst, const void* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          su32(dst)),
      "l"(map), "r"(su32(bar)), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const void* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
          su32(dst)),
      "l"(map), "r"(su32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(bar)) : "memory");
}

// tensor memory
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(dst_smem)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, one CTA, kind::f16
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T: A in tensor memory, row m in lane m, two
// consecutive fp16 of K per 32-bit column
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 16 consecutive 32-bit columns of this warp's 32 lanes, written from registers
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// arrive once on an mbarrier when every MMA issued so far by this thread is done
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
               : "memory");
}
// 16 consecutive 32-bit columns of this warp's 32 lanes (lane i of the warp
// reads tensor-memory lane (taddr >> 16) + i)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
#endif  // __CUDACC__

// tc_plan_kernel: chunks of the bucketed work list
struct TcPlanArgs {
  const int* n_uniq;    // touched experts (work items) of the call
  const int* uniq_e;    // item -> expert id (-1: shared expert)
  const int* uniq_off;  // item -> first entry; [n_uniq] = number of entries
  int bits, shared_bits;
  TcChunk* chunks;      // [max_chunks]
  int* n_chunks;
  int max_chunks;
  WsHeader* hdr;
};

// tc_pack_kernel: B operand rows of every entry
struct TcPackArgs {
  const float* src;     // fp32 rows: per token (by_token) or per (token, slot) id
  int by_token, nslots, K;
  const int* ent;       // entry -> token * nslots + slot
  const int* n_uniq;
  const int* uniq_off;
  int n_ids;            // batch * nslots: (token, slot) ids
  __half* dst;          // [entries * 2][K]: hi row, lo row
  float* scale;         // [entries]: 2^e
  WsHeader* hdr;
};

// tc_contract_kernel: one pass over the units of a call
struct TcContractArgs {
  int mode;             // 0: gate/up (SwiGLU epilogue), 1: down
  int rows;             // weight rows per expert: 2 * inter or hidden
  int ng;               // groups along K
  int tiles;            // ceil(rows / kTcM)
  int out_cols;         // row length of `out` (inter or hidden)
  const TcChunk* chunks;
  const int* n_chunks;
  const int* ent;
  const float* bscale;  // [entries] scale of the B rows
  float* out;           // [(token, slot) id][out_cols]
  int max_entries;      // size of ent / bscale
  int n_ids;            // rows of out: batch * slots
  WsHeader* hdr;
};

// One batched contraction pass of a layer (host side).  The kernels are
// launched by launch_tc_* in stream order: plan, pack(x), contract(gate/up),
// pack(a), contract(down).
struct TcLaunch {
  int H, I, E, bits, shared_bits, has_shared;
  const uint8_t* experts;  // pool of packed experts, `stride` bytes apart
  size_t stride;
  const uint8_t* shared;
  const TcChunk* chunks;   // work list (tc_plan_kernel)
  const int* n_chunks;
  int max_chunks;
  const int* ent;          // bucketed entries
  int max_entries;
  const __half* xops;      // [max_entries * 2][H] B rows of the hidden states
  const float* xscale;
  const __half* aops;      // [max_entries * 2][I] B rows of the activations
  const float* ascale;
  float* a_out;            // [(token, slot) id][I] SwiGLU activations
  float* d_out;            // [(token, slot) id][H] expert outputs
  WsHeader* hdr;
};
bool tc_supported(const TcLaunch& L);
cudaError_t launch_tc_single_item(int B, int* n_uniq, int* uniq_e, int* uniq_off, int* ent, cudaStream_t s);
cudaError_t launch_tc_plan(const TcPlanArgs& a, cudaStream_t s);
cudaError_t launch_tc_pack(const TcPackArgs& a, int max_entries, cudaStream_t s);
cudaError_t launch_tc_contract(const TcLaunch& L, int mode, cudaStream_t s);

}  // namespace tc
}  // namespace moe
