// Internal declarations shared by the kernel files and the C-ABI layer.
#pragma once

#include <algorithm>
#include <atomic>
#include <cstddef>
#include <string>
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "moe_device.cuh"

namespace moe {

constexpr int kBlock = 512;   // threads per block of the matvec kernels
constexpr int kWarps = kBlock / 32;
constexpr int kSharedChunk = 32;  // batched path: shared-expert tokens per work item


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
  uint8_t* q;   // limb vectors [rows][ng * kLimbBytes]
  float2* e;    // [rows][ng]
  WsHeader* hdr;
};

struct RouterArgs {
  const float* xn;
  int B, H, E;
  int stages_per_split;  // router_stages_per_split(B, H, E)
  const uint16_t* router;
  const uint16_t* gate;  // extra row E, or null
  float* logits;         // partial sums [splits][B][E + 1]
};

struct TopkArgs {
  const float* logits;  // router partial sums [splits][B][E + 1]
  const float* offset;  // [B, E] or null
  int B, splits;
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
  const uint8_t* xq;   // limbs of each token's xn
  const float2* xe;
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
  const uint8_t* aq;   // limbs of each (token, slot) activation
  const float2* ae;
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

// Shared-memory plan of the single-token kernel (byte offsets into dynamic smem).
struct DecodePlan {
  int P;            // grid size: one block per SM
  int rows_gu;      // max gate/up row pairs per block
  int rows_d;       // max down rows per block
  int rows_r;       // max router rows per block (incl. the shared-gate row)
  int part_stride;  // floats per gate/up partial buffer
  size_t gu_slot;   // bytes of one routed expert's gate/up slice
  size_t dn_slot;   // bytes of one expert's down slice
  size_t off_dn;    // down slices, slot p at off_dn + p * dn_slot
  size_t off_g;     // gate/up area (before routing: shared slice, router rows)
  size_t off_sgu, off_rt, off_hbuf;  // relative to off_g, before routing
  size_t off_pdn;   // relative to off_g: down partials, after the gate/up phase
  size_t off_al, off_ae;   // limbs of x, later of every expert's activation
  size_t off_part, off_rpart, off_y, off_bar, off_misc;
  size_t total;
};

// The weights and per-layer outputs of one layer (9 words: the stack kernel
// copies them into shared memory word by word).
struct DecodeLayer {
  const uint8_t* experts;
  size_t stride;
  const uint8_t* shared;
  const uint16_t* router;
  const uint16_t* gamma;
  const uint16_t* gate;
  const float* offset;
  int32_t* idx_out;
  float* w_out;
};
static_assert(sizeof(DecodeLayer) == 72, "DecodeLayer is copied as 9 words");

struct DecodeArgs {
  int H, I, E, K, bits, shared_bits, has_shared, has_gate;
  float eps;
  float* h;
  WsHeader* hdr;
  unsigned long long* pub_logits;  // [E + 1] published words
  unsigned long long* pub_act;     // [(K + 1), I] published words (weighted activations)
  DecodePlan plan;
  DecodeLayer ly;                  // the layer (single-layer kernel)
};

// Layers of one token in one launch of the single-token kernel: layer l's
// output is layer l + 1's input.  Every layer has the shape and code widths
// of d; d.ly is unused.
constexpr int kMaxStackLayers = 64;
struct StackArgs {
  DecodeArgs d;
  unsigned long long* pub_h;  // [H rounded up to 128] published words: a layer's output rows
  int L;
  DecodeLayer layers[kMaxStackLayers];
};

cudaError_t launch_pack(const PackArgs& a, cudaStream_t s);
cudaError_t launch_norm_quant(const NormQuantArgs& a, int B, cudaStream_t s);
// Router splits of the input dimension: a function of the shape only.
int router_splits(int B, int H, int E);
int router_stages_per_split(int B, int H, int E);
cudaError_t launch_router(const RouterArgs& a, cudaStream_t s);
cudaError_t launch_topk(const TopkArgs& a, int B, cudaStream_t s);
cudaError_t launch_bucket(const BucketArgs& a, cudaStream_t s);
cudaError_t launch_gateup(const GateUpArgs& a, int items, cudaStream_t s);
cudaError_t launch_down(const DownArgs& a, int items, cudaStream_t s);
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s);

// Single-token layer: plan (false when the shape does not fit) and launch.
bool decode_plan(int H, int I, int E, int K, int bits, int shared_bits, int has_shared, int has_gate, int device,
                 DecodePlan* out);
bool decode_plan_for(int nsm, int optin, int H, int I, int E, int K, int bits, int shared_bits, int has_shared,
                     int has_gate, DecodePlan* out);
cudaError_t launch_decode(const DecodeArgs& a, bool pdl, cudaStream_t s);
cudaError_t launch_decode_stack(const StackArgs& a, bool pdl, cudaStream_t s);

// Launches of the multi-kernel path.  Inside a PdlScope that is on, kernels go
// out with programmatic stream serialisation: each may be scheduled while its
// predecessor on the stream drains, and every such kernel starts with
// griddepcontrol.wait (pdl_wait_prior) before it touches memory, so the
// ordering of the stream is kept; the gain is the launch latency between the
// short kernels of a batched call.
extern thread_local bool t_launch_pdl;
struct PdlScope {
  bool prev;
  explicit PdlScope(bool on) : prev(t_launch_pdl) { t_launch_pdl = on; }
  ~PdlScope() { t_launch_pdl = prev; }
};
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (t_launch_pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Text returned by moe_last_error_message() for this thread.
void set_last_error(const std::string& msg);

// Opt-in dynamic shared memory of a kernel, raised once per device to the
// largest size launched so far (the attribute is per device; calls from
// several threads at once only repeat the same setting).
constexpr int kMaxDevices = 64;
template <typename Kernel>
cudaError_t ensure_dynamic_smem(Kernel kernel, int bytes, std::atomic<int> (&configured)[kMaxDevices]) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (configured[dev].load(std::memory_order_relaxed) >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) configured[dev].store(bytes, std::memory_order_relaxed);
  return e;
}

}  // namespace moe
