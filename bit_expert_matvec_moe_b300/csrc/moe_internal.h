// Internal declarations shared by the kernel files and the C-ABI layer.
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "moe_device.cuh"

namespace moe {

constexpr int kBlock = 512;   // threads per block of the matvec kernels
constexpr int kRowsGU = 8;    // gate/up row pairs per block (multi-kernel path)
constexpr int kRowsD = 32;    // down rows per block (multi-kernel path)
constexpr int kMaxSlots = 3;  // gate/up staging ring of the fused kernel

struct PackArgs {
  Fmt f;
  const uint8_t* codes[3];
  const uint16_t* scales[3];
  const uint16_t* biases[3];
  uint8_t* dst;
};

struct NormQuantArgs {
  const float* in;
  int n;
  int do_norm;
  float eps;
  const uint16_t* gamma;
  float* xn_out;
  int layouts;  // bit 0: 4-bit limb order, bit 1: 2-bit limb order
  uint32_t* q4;
  float2* e4;
  uint32_t* q2;
  float2* e2;
  WsHeader* hdr;
};

struct RouterArgs {
  const float* xn;
  int B, H, E;
  const uint16_t* router;
  const uint16_t* gate;  // extra row E, or null
  const float* offset;   // [B, E] or null
  float* logits;         // [B, E + 1]
};

struct TopkArgs {
  const float* logits;  // [B, E + 1]
  int E, K, has_gate;
  int32_t* idx;
  float* w;
  float* gs;
  int32_t* idx_out;
  float* w_out;
  float* logits_out;
  WsHeader* hdr;
};

struct BucketArgs {
  const int32_t* idx;
  int B, K, E, has_shared, nslots;
  int* n_uniq;
  int* uniq_e;    // [E + 1]
  int* uniq_off;  // [E + 2]
  int* ent;       // [B * nslots]
};

struct GateUpArgs {
  int H, I, K, B, nslots;
  int bits, shared_bits;
  const uint8_t* experts;
  size_t stride;
  const uint8_t* shared;
  const uint8_t* blob;  // single-expert mode when uniq_e == null
  const int* n_uniq;
  const int* uniq_e;
  const int* uniq_off;
  const int* ent;
  const uint32_t* xq4;
  const float2* xe4;
  const uint32_t* xq2;
  const float2* xe2;
  float* a_out;  // [B * nslots, I]
};

struct DownArgs {
  int H, I, K, B, nslots;
  int bits, shared_bits;
  const uint8_t* experts;
  size_t stride;
  const uint8_t* shared;
  const uint8_t* blob;
  const int* n_uniq;
  const int* uniq_e;
  const int* uniq_off;
  const int* ent;
  const uint32_t* aq4;
  const float2* ae4;
  const uint32_t* aq2;
  const float2* ae2;
  float* d_out;  // [B * nslots, H]
};

struct CombineArgs {
  int B, H, K, nslots, has_shared, single, accumulate;
  const float* d;
  const float* w;
  const float* gs;
  const float* row_w;
  float* out;
};

// Shared-memory plan of the fused single-token kernel (byte offsets).
struct FusedPlan {
  int P;           // grid size (co-resident blocks)
  int nslots;      // gate/up staging slots
  int rows_gu;     // max gate/up row pairs per block
  int rows_d;      // max down rows per block
  size_t slot_bytes;
  size_t off_x, off_xq4, off_xq2, off_xe4, off_xe2, off_ae, off_gu, off_dn[kMaxTopK + 1], off_part, off_pd,
      off_logits, off_bar, total;
};

struct FusedArgs {
  int H, I, E, K, bits, shared_bits, has_shared, has_gate;
  float eps;
  const uint8_t* experts;
  size_t stride;
  const uint8_t* shared;
  const uint16_t* router;
  const uint16_t* gamma;
  const uint16_t* gate;
  float* h;
  const float* offset;
  int32_t* idx_out;
  float* w_out;
  WsHeader* hdr;
  float* a_glob;   // [(K + 1), I]
  float* logits;   // [E + 1]
  FusedPlan plan;
};

cudaError_t launch_pack(const PackArgs& a, cudaStream_t s);
cudaError_t launch_norm_quant(const NormQuantArgs& a, int B, cudaStream_t s);
cudaError_t launch_router(const RouterArgs& a, cudaStream_t s);
cudaError_t launch_topk(const TopkArgs& a, int B, cudaStream_t s);
cudaError_t launch_bucket(const BucketArgs& a, cudaStream_t s);
cudaError_t launch_gateup(const GateUpArgs& a, int items, cudaStream_t s);
cudaError_t launch_down(const DownArgs& a, int items, cudaStream_t s);
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s);

// Fused single-token layer: plan (false when the shape does not fit) and launch.
bool fused_plan(int H, int I, int E, int K, int bits, int shared_bits, int has_shared, int device, FusedPlan* out);
cudaError_t launch_fused(const FusedArgs& a, cudaStream_t s);

}  // namespace moe
