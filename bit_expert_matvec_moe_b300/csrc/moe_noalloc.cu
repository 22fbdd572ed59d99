// moe_layer_decode_noalloc: the single-token layer for callers that cannot
// allocate device memory.  Some callers run where no allocator is available to
// them: code inside another framework's memory pool that must not call
// cudaMalloc, a stream-ordered pipeline that forbids allocation on its hot
// path, or a plugin that is handed only its input and output buffers.  They
// cannot provide the workspace that moe_layer_decode needs, so this entry point
// keeps that workspace in a fixed array of device memory that the library owns.
//
// The array is a file-scope static __device__ symbol; every GPU that loads the
// library holds it until the process exits.  Host code cannot use the symbol's
// name as a device address: the address is fetched with cudaGetSymbolAddress
// on each call, with the caller's device current.
#include <mutex>
#include <string>

#include "../../include/moe.h"
#include <cstddef>

#include "moe_internal.h"

using namespace moe;

namespace {

constexpr size_t kScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;

// header, then published logits, then published activations (the single-token
// kernel's cross-block state); zeroed once per device at set-up
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};
thread_local bool t_test_timeout_next = false;  // moe_noalloc_test_timeout_next

moe_status fail(cudaError_t e, const char* what) {
  set_last_error(std::string(what) + ": " + cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}

// Device address of the scratch array on `dev` (current).  The address is
// looked up on every call (cheap), so that a module reloaded after a device
// reset is noticed; whenever it differs from the one seen before on this
// device, the whole array is cleared on `s` first (the launch counters and the
// epoch words of published results must start together at zero).  The clear
// is stream-ordered: it synchronises nothing else on the device.
moe_status scratch_for(int dev, cudaStream_t s, void** out) {
  if (dev < 0 || dev >= kMaxDevices) {
    set_last_error("device index out of range");
    return MOE_ERR_UNSUPPORTED;
  }
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
  if (e != cudaSuccess) return fail(e, "cudaGetSymbolAddress");
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] != p) {
    e = cudaMemsetAsync(p, 0, kScratchBytes, s);
    if (e != cudaSuccess) return fail(e, "clearing the scratch array");
    g_addr[dev] = p;
  }
  *out = p;
  return MOE_OK;
}

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" {

moe_status moe_layer_decode_noalloc(const moe_layer* layer, float* h, const float* logit_offset, int32_t* idx_out,
                                    float* w_out, int32_t* status_out, moe_stream_t stream) {
  if (!layer || !h || !layer->experts || !layer->router) return MOE_ERR_INVALID_ARG;
  const moe_dims& d = layer->d;
  if (d.group != MOE_GROUP || (d.bits != 4 && d.bits != 2)) return MOE_ERR_INVALID_ARG;
  if (d.hidden <= 0 || d.hidden % MOE_GROUP || d.inter <= 0 || d.inter % MOE_GROUP || d.n_experts < 1 ||
      d.top_k < 1 || d.top_k > MOE_MAX_TOPK || d.top_k > d.n_experts || !(d.rms_eps >= 0.f))
    return MOE_ERR_INVALID_ARG;
  if (d.flags & ~(MOE_HAS_SHARED | MOE_HAS_SHARED_GATE | MOE_PDL)) return MOE_ERR_INVALID_ARG;
  const int has_shared = (d.flags & MOE_HAS_SHARED) ? 1 : 0;
  const int has_gate = (d.flags & MOE_HAS_SHARED_GATE) ? 1 : 0;
  if (has_gate && (!has_shared || !layer->shared_gate)) return MOE_ERR_INVALID_ARG;
  if (has_shared && (!layer->shared || (layer->shared_bits != 4 && layer->shared_bits != 2))) return MOE_ERR_INVALID_ARG;
  const size_t blob = make_fmt(d.bits, d.hidden, d.inter).total;
  if (layer->expert_stride < blob || layer->expert_stride % 16) return MOE_ERR_INVALID_ARG;
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!a16(h) || !a16(layer->experts) || !a16(layer->router) || (has_shared && !a16(layer->shared)) ||
      (layer->rms_gamma && !a16(layer->rms_gamma)) || (has_gate && !a16(layer->shared_gate)) ||
      (logit_offset && !a16(logit_offset)) || (idx_out && !a16(idx_out)) || (w_out && !a16(w_out)) ||
      !status_out || (reinterpret_cast<uintptr_t>(status_out) & 3u))
    return MOE_ERR_INVALID_ARG;

  // sizes: the scratch holds the header, E + 1 published logits and
  // (K + 1) * inter published activations (8 bytes each)
  const size_t off_logits = 256;
  const size_t off_act = off_logits + up256((size_t)(d.n_experts + 1) * 8);
  const size_t need = off_act + up256((size_t)(d.top_k + 1) * d.inter * 8);
  if (need > kScratchBytes) {
    set_last_error("layer too large for the fixed scratch array: needs " + std::to_string(need) +
                   " bytes, holds " + std::to_string(kScratchBytes));
    return MOE_ERR_UNSUPPORTED;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(e, "cudaGetDevice");
  const int shared_bits = has_shared ? layer->shared_bits : d.bits;
  DecodePlan plan;
  if (!decode_plan(d.hidden, d.inter, d.n_experts, d.top_k, d.bits, shared_bits, has_shared, has_gate, dev, &plan)) {
    set_last_error("shape outside the single-token kernel (hidden <= 4096, inter <= 2048, shared memory plan)");
    return MOE_ERR_UNSUPPORTED;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  moe_status st = scratch_for(dev, s, &scratch);
  if (st != MOE_OK) return st;
  uint8_t* base = static_cast<uint8_t*>(scratch);

  // each call starts with a clear error state (the launch counters live on)
  e = cudaMemsetAsync(base, 0, kHeaderErrorBytes, s);
  if (e != cudaSuccess) return fail(e, "cudaMemsetAsync");
  if (t_test_timeout_next) {
    // test hook, one call: every cross-block wait of this launch expects a
    // later epoch (header bar_extra = 1), so each block gives up after its
    // bounded wait and the call reports a timeout
    t_test_timeout_next = false;
    e = cudaMemsetAsync(base + offsetof(WsHeader, bar_extra), 1, 1, s);
    if (e != cudaSuccess) return fail(e, "cudaMemsetAsync");
  }

  DecodeArgs f{};
  f.H = d.hidden;
  f.I = d.inter;
  f.E = d.n_experts;
  f.K = d.top_k;
  f.bits = d.bits;
  f.shared_bits = shared_bits;
  f.has_shared = has_shared;
  f.has_gate = has_gate;
  f.eps = d.rms_eps;
  f.ly.experts = static_cast<const uint8_t*>(layer->experts);
  f.ly.stride = layer->expert_stride;
  f.ly.shared = static_cast<const uint8_t*>(layer->shared);
  f.ly.router = layer->router;
  f.ly.gamma = layer->rms_gamma;
  f.ly.gate = layer->shared_gate;
  f.h = h;
  f.ly.offset = logit_offset;
  f.ly.idx_out = idx_out;
  f.ly.w_out = w_out;
  f.hdr = reinterpret_cast<WsHeader*>(base);
  f.pub_logits = reinterpret_cast<unsigned long long*>(base + off_logits);
  f.pub_act = reinterpret_cast<unsigned long long*>(base + off_act);
  f.plan = plan;
  e = launch_decode(f, (d.flags & MOE_PDL) != 0, s);
  if (e != cudaSuccess) return fail(e, "launch");
  // the device status word of this call (0 = ok), copied on the stream: the
  // caller cannot reach the array, and the next call clears it
  e = cudaMemcpyAsync(status_out, base, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) return fail(e, "cudaMemcpyAsync");
  return MOE_OK;
}

moe_status moe_noalloc_test_timeout_next(void) {
  t_test_timeout_next = true;
  return MOE_OK;
}

}  // extern "C"
