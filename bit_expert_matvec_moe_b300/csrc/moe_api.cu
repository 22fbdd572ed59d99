// C ABI of the MoE decode path: argument checks, workspace layout and launches.
// Declarations and their contract: include/moe.h.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <string>

#include "../../include/moe.h"
#include "moe_internal.h"
#include "moe_tc.cuh"

using namespace moe;

// The tensor-core contraction (MOE_TENSOR_CORES) is accepted when this is 1
// (the default); a build with 0 refuses the flag in both entry points that
// take it, with MOE_ERR_UNSUPPORTED.
#ifndef MOE_TC_ENABLED
#define MOE_TC_ENABLED 1
#endif

namespace {

thread_local std::string g_last_error;

bool tc_refused(const moe_dims& d, int B) {
  if (MOE_TC_ENABLED || B <= 1 || !(d.flags & MOE_TENSOR_CORES)) return false;
  g_last_error = "MOE_TENSOR_CORES: the tensor-core contraction is not enabled in this build";
  return true;
}

moe_status cuda_fail(cudaError_t e) {
  g_last_error = cudaGetErrorString(e);
  return MOE_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dims_ok(const moe_dims* d) {
  if (!d) return false;
  if (d->group != MOE_GROUP) return false;
  if (d->hidden <= 0 || d->hidden % MOE_GROUP || d->hidden > MOE_MAX_HIDDEN) return false;
  if (d->inter <= 0 || d->inter % MOE_GROUP || d->inter > MOE_MAX_INTER) return false;
  if (d->n_experts < 1 || d->n_experts > MOE_MAX_EXPERTS) return false;
  if (d->top_k < 1 || d->top_k > MOE_MAX_TOPK || d->top_k > d->n_experts) return false;
  if (d->bits != 4 && d->bits != 2) return false;
  if (!(d->rms_eps >= 0.f) || !std::isfinite(d->rms_eps)) return false;
  if (d->flags & ~(MOE_HAS_SHARED | MOE_HAS_SHARED_GATE | MOE_NO_FUSED | MOE_PDL | MOE_TENSOR_CORES)) return false;
  if ((d->flags & MOE_HAS_SHARED_GATE) && !(d->flags & MOE_HAS_SHARED)) return false;
  return true;
}

struct WsLayout {
  size_t logits, idx, w, gs, xn, xq, xe, a, aq, ae, d, nuniq, uniq_e, uniq_off, ent, pub_logits, pub_act, pub_h;
  // tensor-core contraction (MOE_TENSOR_CORES only): B operand rows and scales, work list
  size_t xops, aops, xscale, ascale, chunks, nchunks;
  int max_chunks;
  size_t total;
};

// Byte offsets of the workspace regions for a batch of B tokens.  Only the
// 256-byte header (status word, launch and exchange counters) lives across
// calls.
WsLayout ws_layout(const moe_dims& d, int B) {
  WsLayout L{};
  size_t o = kHeaderBytes;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = (o + bytes + 255) & ~size_t(255);
    return at;
  };
  const size_t E = d.n_experts, K = d.top_k, H = d.hidden, I = d.inter;
  const size_t ns = K + 1;  // routed slots plus the shared slot
  const size_t ngh = H / MOE_GROUP, ngi = I / MOE_GROUP;
  // the single-token kernel's published words first, at offsets that do not
  // depend on the batch (epoch << 32 | value)
  L.pub_logits = take((size_t)(MOE_MAX_EXPERTS + 1) * 8);
  L.pub_act = take(ns * I * 8);
  L.pub_h = take((H + 127) / 128 * 128 * 8);  // a stack launch's layer outputs (slots in chunks of 128)
  L.logits = take((size_t)router_splits(B, (int)H, (int)E) * B * (E + 1) * 4);
  L.idx = take(B * K * 4);
  L.w = take(B * K * 4);
  L.gs = take(B * 4);
  L.xn = take(B * H * 4);
  L.xq = take(B * ngh * kLimbBytes);
  L.xe = take(B * ngh * 8);
  L.a = take(B * ns * I * 4);
  L.aq = take(B * ns * ngi * kLimbBytes);
  L.ae = take(B * ns * ngi * 8);
  L.d = take(B * ns * H * 4);
  L.nuniq = take(4);
  const size_t shared_items = (B + kSharedChunk - 1) / kSharedChunk;  // the shared expert's work items
  L.uniq_e = take((E + shared_items) * 4);
  L.uniq_off = take((E + shared_items + 1) * 4);
  L.ent = take(B * ns * 4);
  if (d.flags & MOE_TENSOR_CORES) {
    const size_t ne = B * ns;  // entries: (token, slot) pairs
    L.xops = take(ne * 2 * H * 2);
    L.aops = take(ne * 2 * I * 2);
    L.xscale = take(ne * 4);
    L.ascale = take(ne * 4);
    // sum over items of ceil(n / kTcTok) <= items + entries / kTcTok
    L.max_chunks = (int)(std::min(B * K, E) + shared_items + (ne + tc::kTcTok - 1) / tc::kTcTok);
    L.chunks = take((size_t)L.max_chunks * sizeof(tc::TcChunk));
    L.nchunks = take(4);
  }
  L.total = o;
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

int current_device() {
  int dev = 0;
  cudaGetDevice(&dev);
  return dev;
}

// The tensor-core contraction of a bucketed work list: plan (chunks of at
// most 32 entries) -> B rows of xn -> gate/up contraction with SwiGLU -> B
// rows of the activations -> down contraction into the workspace's d rows.
struct TcSource {
  const uint8_t* experts;
  size_t stride;
  int E, bits;
  const uint8_t* shared;
  int shared_bits, has_shared;
  const float* xn;  // [tokens][H]
};
moe_status run_tc(const moe_dims& d, const WsLayout& L, void* ws, int B, int nslots, const TcSource& src,
                  int* n_uniq, int* uniq_e, int* uniq_off, int* ent, cudaStream_t s) {
  WsHeader* hdr = at<WsHeader>(ws, 0);
  tc::TcLaunch tl{};
  tl.H = d.hidden;
  tl.I = d.inter;
  tl.E = src.E;
  tl.bits = src.bits;
  tl.shared_bits = src.shared_bits;
  tl.has_shared = src.has_shared;
  tl.experts = src.experts;
  tl.stride = src.stride;
  tl.shared = src.shared;
  tl.chunks = at<tc::TcChunk>(ws, L.chunks);
  tl.n_chunks = at<int>(ws, L.nchunks);
  tl.max_chunks = L.max_chunks;
  tl.ent = ent;
  tl.max_entries = B * nslots;
  tl.xops = at<__half>(ws, L.xops);
  tl.xscale = at<float>(ws, L.xscale);
  tl.aops = at<__half>(ws, L.aops);
  tl.ascale = at<float>(ws, L.ascale);
  tl.a_out = at<float>(ws, L.a);
  tl.d_out = at<float>(ws, L.d);
  tl.hdr = hdr;
  if (!tc::tc_supported(tl)) {
    set_last_error("MOE_TENSOR_CORES: layer layout not supported by the tensor-core contraction");
    return MOE_ERR_UNSUPPORTED;
  }
  cudaError_t e;
  tc::TcPlanArgs pl{};
  pl.n_uniq = n_uniq;
  pl.uniq_e = uniq_e;
  pl.uniq_off = uniq_off;
  pl.bits = src.bits;
  pl.shared_bits = src.shared_bits;
  pl.chunks = at<tc::TcChunk>(ws, L.chunks);
  pl.n_chunks = at<int>(ws, L.nchunks);
  pl.max_chunks = L.max_chunks;
  pl.hdr = hdr;
  if ((e = tc::launch_tc_plan(pl, s)) != cudaSuccess) return cuda_fail(e);
  tc::TcPackArgs px{};
  px.src = src.xn;
  px.by_token = 1;
  px.nslots = nslots;
  px.K = d.hidden;
  px.ent = ent;
  px.n_uniq = n_uniq;
  px.uniq_off = uniq_off;
  px.n_ids = B * nslots;
  px.dst = at<__half>(ws, L.xops);
  px.scale = at<float>(ws, L.xscale);
  px.hdr = hdr;
  if ((e = tc::launch_tc_pack(px, B * nslots, s)) != cudaSuccess) return cuda_fail(e);
  if ((e = tc::launch_tc_contract(tl, 0, s)) != cudaSuccess) return cuda_fail(e);
  tc::TcPackArgs pa = px;
  pa.src = tl.a_out;
  pa.by_token = 0;
  pa.K = d.inter;
  pa.dst = at<__half>(ws, L.aops);
  pa.scale = at<float>(ws, L.ascale);
  if ((e = tc::launch_tc_pack(pa, B * nslots, s)) != cudaSuccess) return cuda_fail(e);
  if ((e = tc::launch_tc_contract(tl, 1, s)) != cudaSuccess) return cuda_fail(e);
  return MOE_OK;
}

}  // namespace

namespace moe {
void set_last_error(const std::string& msg) { g_last_error = msg; }
}  // namespace moe

extern "C" {

size_t moe_packed_expert_bytes(const moe_dims* dims, int32_t bits) {
  if (!dims_ok(dims) || (bits != 4 && bits != 2)) return 0;
  return make_fmt(bits, dims->hidden, dims->inter).total;
}

size_t moe_workspace_bytes(const moe_dims* dims, int32_t max_batch) {
  if (!dims_ok(dims) || max_batch < 1 || max_batch > MOE_MAX_BATCH) return 0;
  return ws_layout(*dims, max_batch).total;
}

moe_status moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!ws || !aligned16(ws) || ws_bytes < kHeaderBytes) return MOE_ERR_INVALID_ARG;
  cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status moe_pack_weights(const moe_dims* dims, int32_t bits, const uint8_t* const codes[3],
                            const uint16_t* const scales[3], const uint16_t* const biases[3], void* dst,
                            moe_stream_t stream) {
  if (!dims_ok(dims) || (bits != 4 && bits != 2) || !codes || !scales || !biases || !dst || !aligned16(dst))
    return MOE_ERR_INVALID_ARG;
  PackArgs a{};
  a.f = make_fmt(bits, dims->hidden, dims->inter);
  for (int m = 0; m < 3; ++m) {
    if (!codes[m] || !scales[m] || !biases[m]) return MOE_ERR_INVALID_ARG;
    if (!aligned16(codes[m]) || (reinterpret_cast<uintptr_t>(scales[m]) & 1u) ||
        (reinterpret_cast<uintptr_t>(biases[m]) & 1u))
      return MOE_ERR_INVALID_ARG;
    a.codes[m] = codes[m];
    a.scales[m] = scales[m];
    a.biases[m] = biases[m];
  }
  a.dst = static_cast<uint8_t*>(dst);
  cudaError_t e = launch_pack(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status moe_route(const moe_dims* dims, const float* xn, int32_t B, const uint16_t* router,
                     const float* logit_offset, int32_t* idx, float* w, float* logits_out, void* ws, size_t ws_bytes,
                     moe_stream_t stream) {
  if (!dims_ok(dims) || B < 1 || B > MOE_MAX_BATCH) return MOE_ERR_INVALID_ARG;
  if (!xn || !router || !idx || !w || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned16(xn) || !aligned16(router) || !aligned16(ws) || !aligned16(idx) || !aligned16(w) ||
      (logit_offset && !aligned16(logit_offset)) || (logits_out && !aligned16(logits_out)))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*dims, B);
  if (ws_bytes < L.total) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PdlScope pdl_scope((dims->flags & MOE_PDL) != 0);
  RouterArgs r{};
  r.xn = xn;
  r.B = B;
  r.H = dims->hidden;
  r.E = dims->n_experts;
  r.router = router;
  r.gate = nullptr;
  r.stages_per_split = router_stages_per_split(B, r.H, r.E);
  r.logits = at<float>(ws, L.logits);
  cudaError_t e = launch_router(r, s);
  if (e != cudaSuccess) return cuda_fail(e);
  TopkArgs t{};
  t.logits = r.logits;
  t.offset = logit_offset;
  t.B = B;
  t.splits = router_splits(B, r.H, r.E);
  t.E = dims->n_experts;
  t.K = dims->top_k;
  t.has_gate = 0;
  t.idx = idx;
  t.w = w;
  t.gs = nullptr;
  t.logits_out = logits_out;
  t.hdr = at<WsHeader>(ws, 0);
  e = launch_topk(t, B, s);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status moe_expert_forward(const moe_dims* dims, int32_t bits, const void* blob, const float* xn, int32_t B,
                              const float* row_w, float* out, int32_t accumulate, void* ws, size_t ws_bytes,
                              moe_stream_t stream) {
  if (!dims_ok(dims) || (bits != 4 && bits != 2) || B < 1 || B > MOE_MAX_BATCH) return MOE_ERR_INVALID_ARG;
  if (!blob || !xn || !out || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned16(blob) || !aligned16(xn) || !aligned16(out) || !aligned16(ws) || (row_w && !aligned16(row_w)))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*dims, B);
  if (ws_bytes < L.total) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PdlScope pdl_scope((dims->flags & MOE_PDL) != 0);
  const int H = dims->hidden, I = dims->inter;
  WsHeader* hdr = at<WsHeader>(ws, 0);
  if (tc_refused(*dims, B)) return MOE_ERR_UNSUPPORTED;
  if (B > 1 && (dims->flags & MOE_TENSOR_CORES)) {
    // one expert for tokens 0 .. B-1: a single work item through the shared-expert maps
    const size_t blob_bytes = make_fmt(bits, H, I).total;
    cudaError_t e = tc::launch_tc_single_item(B, at<int>(ws, L.nuniq), at<int>(ws, L.uniq_e), at<int>(ws, L.uniq_off),
                                              at<int>(ws, L.ent), s);
    if (e != cudaSuccess) return cuda_fail(e);
    TcSource src{};
    src.experts = static_cast<const uint8_t*>(blob);
    src.stride = blob_bytes;
    src.E = 1;
    src.bits = bits;
    src.shared = static_cast<const uint8_t*>(blob);
    src.shared_bits = bits;
    src.has_shared = 1;
    src.xn = xn;
    const moe_status st =
        run_tc(*dims, L, ws, B, 1, src, at<int>(ws, L.nuniq), at<int>(ws, L.uniq_e), at<int>(ws, L.uniq_off),
               at<int>(ws, L.ent), s);
    if (st != MOE_OK) return st;
    CombineArgs cb{};
    cb.B = B;
    cb.H = H;
    cb.K = 0;
    cb.nslots = 1;
    cb.single = 1;
    cb.accumulate = accumulate ? 1 : 0;
    cb.d = at<float>(ws, L.d);
    cb.row_w = row_w;
    cb.out = out;
    e = launch_combine(cb, s);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e);
  }
  NormQuantArgs nq{};
  nq.in = xn;
  nq.n = H;
  nq.do_norm = 0;
  nq.q = at<uint8_t>(ws, L.xq);
  nq.e = at<float2>(ws, L.xe);
  nq.hdr = hdr;
  cudaError_t e = launch_norm_quant(nq, B, s);
  if (e != cudaSuccess) return cuda_fail(e);

  GateUpArgs g{};
  g.H = H;
  g.I = I;
  g.K = 0;
  g.B = B;
  g.nslots = 1;
  g.bits = bits;
  g.shared_bits = bits;
  g.blob = static_cast<const uint8_t*>(blob);
  g.xq = nq.q;
  g.xe = nq.e;
  g.a_out = at<float>(ws, L.a);
  e = launch_gateup(g, 1, s);
  if (e != cudaSuccess) return cuda_fail(e);

  NormQuantArgs aq = nq;
  aq.in = g.a_out;
  aq.n = I;
  aq.q = at<uint8_t>(ws, L.aq);
  aq.e = at<float2>(ws, L.ae);
  e = launch_norm_quant(aq, B, s);
  if (e != cudaSuccess) return cuda_fail(e);

  DownArgs dn{};
  dn.H = H;
  dn.I = I;
  dn.K = 0;
  dn.B = B;
  dn.nslots = 1;
  dn.bits = bits;
  dn.shared_bits = bits;
  dn.blob = g.blob;
  dn.aq = aq.q;
  dn.ae = aq.e;
  dn.d_out = at<float>(ws, L.d);
  e = launch_down(dn, 1, s);
  if (e != cudaSuccess) return cuda_fail(e);

  CombineArgs cb{};
  cb.B = B;
  cb.H = H;
  cb.K = 0;
  cb.nslots = 1;
  cb.single = 1;
  cb.accumulate = accumulate ? 1 : 0;
  cb.d = at<float>(ws, L.d);
  cb.row_w = row_w;
  cb.out = out;
  e = launch_combine(cb, s);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

// A layer's own buffers and dims (the checks every layer call makes).
static bool layer_ok(const moe_layer* layer) {
  if (!layer || !dims_ok(&layer->d)) return false;
  const moe_dims& d = layer->d;
  const int has_shared = (d.flags & MOE_HAS_SHARED) ? 1 : 0;
  const int has_gate = (d.flags & MOE_HAS_SHARED_GATE) ? 1 : 0;
  if (!layer->experts || !layer->router) return false;
  if (has_shared && (!layer->shared || (layer->shared_bits != 4 && layer->shared_bits != 2))) return false;
  if (has_gate && !layer->shared_gate) return false;
  const size_t blob = make_fmt(d.bits, d.hidden, d.inter).total;
  if (layer->expert_stride < blob || layer->expert_stride % 16) return false;
  return aligned16(layer->experts) && aligned16(layer->router) && (!has_shared || aligned16(layer->shared)) &&
         (!layer->rms_gamma || aligned16(layer->rms_gamma)) && (!has_gate || aligned16(layer->shared_gate));
}

// The single-token kernel's pointers of one layer.
static DecodeLayer decode_layer_of(const moe_layer& layer, const float* logit_offset, int32_t* idx_out, float* w_out) {
  DecodeLayer y{};
  y.experts = static_cast<const uint8_t*>(layer.experts);
  y.stride = layer.expert_stride;
  y.shared = static_cast<const uint8_t*>(layer.shared);
  y.router = layer.router;
  y.gamma = layer.rms_gamma;
  y.gate = layer.shared_gate;
  y.offset = logit_offset;
  y.idx_out = idx_out;
  y.w_out = w_out;
  return y;
}

// The single-token kernel's arguments (no layer) when the shape fits it.
static bool decode_args_for(const moe_dims& d, int shared_bits, float* h, void* ws, const WsLayout& L, DecodeArgs* f) {
  const int has_shared = (d.flags & MOE_HAS_SHARED) ? 1 : 0;
  const int has_gate = (d.flags & MOE_HAS_SHARED_GATE) ? 1 : 0;
  if (d.flags & MOE_NO_FUSED) return false;
  DecodePlan plan;
  if (!decode_plan(d.hidden, d.inter, d.n_experts, d.top_k, d.bits, shared_bits, has_shared, has_gate,
                   current_device(), &plan))
    return false;
  *f = DecodeArgs{};
  f->H = d.hidden;
  f->I = d.inter;
  f->E = d.n_experts;
  f->K = d.top_k;
  f->bits = d.bits;
  f->shared_bits = shared_bits;
  f->has_shared = has_shared;
  f->has_gate = has_gate;
  f->eps = d.rms_eps;
  f->h = h;
  f->hdr = at<WsHeader>(ws, 0);
  f->pub_logits = at<unsigned long long>(ws, L.pub_logits);
  f->pub_act = at<unsigned long long>(ws, L.pub_act);
  f->plan = plan;
  return true;
}

static moe_status layer_decode_checked(const moe_layer* layer, float* h, int32_t B, const float* logit_offset,
                                       int32_t* idx_out, float* w_out, void* ws, size_t ws_bytes,
                                       moe_stream_t stream);

moe_status moe_layer_decode(const moe_layer* layer, float* h, int32_t B, const float* logit_offset, int32_t* idx_out,
                            float* w_out, void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!layer_ok(layer) || B < 1 || B > MOE_MAX_BATCH) return MOE_ERR_INVALID_ARG;
  if (!h || !ws || !aligned16(h) || !aligned16(ws) || (logit_offset && !aligned16(logit_offset)) ||
      (idx_out && !aligned16(idx_out)) || (w_out && !aligned16(w_out)))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < ws_layout(layer->d, B).total) return MOE_ERR_INVALID_ARG;
  return layer_decode_checked(layer, h, B, logit_offset, idx_out, w_out, ws, ws_bytes, stream);
}

moe_status moe_stack_decode(const moe_layer* layers, int32_t n_layers, float* h, const float* logit_offset,
                            int32_t* idx_out, float* w_out, void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!layers || n_layers < 1 || !layer_ok(&layers[0])) return MOE_ERR_INVALID_ARG;
  const moe_dims& d = layers[0].d;
  const int has_shared = (d.flags & MOE_HAS_SHARED) ? 1 : 0;
  for (int l = 1; l < n_layers; ++l) {
    const moe_dims& o = layers[l].d;
    if (!layer_ok(&layers[l]) || o.hidden != d.hidden || o.inter != d.inter || o.n_experts != d.n_experts ||
        o.top_k != d.top_k || o.group != d.group || o.bits != d.bits || o.rms_eps != d.rms_eps ||
        o.flags != d.flags || (has_shared && layers[l].shared_bits != layers[0].shared_bits))
      return MOE_ERR_INVALID_ARG;
  }
  // the per-layer rows of the offsets and outputs are read and written one
  // element at a time: 4-byte alignment
  auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (!h || !ws || !aligned16(h) || !aligned16(ws) || (logit_offset && !a4(logit_offset)) ||
      (idx_out && !a4(idx_out)) || (w_out && !a4(w_out)))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(d, 1);
  if (ws_bytes < L.total) return MOE_ERR_INVALID_ARG;
  const int E = d.n_experts, K = d.top_k;
  auto row_off = [&](int l) { return logit_offset ? logit_offset + (size_t)l * E : nullptr; };
  auto row_idx = [&](int l) { return idx_out ? idx_out + (size_t)l * K : nullptr; };
  auto row_w = [&](int l) { return w_out ? w_out + (size_t)l * K : nullptr; };
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  StackArgs sa{};
  if (decode_args_for(d, has_shared ? layers[0].shared_bits : d.bits, h, ws, L, &sa.d)) {
    sa.pub_h = at<unsigned long long>(ws, L.pub_h);
    for (int l0 = 0; l0 < n_layers; l0 += kMaxStackLayers) {
      sa.L = std::min(kMaxStackLayers, n_layers - l0);
      for (int i = 0; i < sa.L; ++i)
        sa.layers[i] = decode_layer_of(layers[l0 + i], row_off(l0 + i), row_idx(l0 + i), row_w(l0 + i));
      const cudaError_t e = launch_decode_stack(sa, (d.flags & MOE_PDL) != 0, s);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    return MOE_OK;
  }
  for (int l = 0; l < n_layers; ++l) {
    const moe_status st = layer_decode_checked(&layers[l], h, 1, row_off(l), row_idx(l), row_w(l), ws, ws_bytes, stream);
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}

// moe_layer_decode after its argument checks.
static moe_status layer_decode_checked(const moe_layer* layer, float* h, int32_t B, const float* logit_offset,
                                       int32_t* idx_out, float* w_out, void* ws, size_t ws_bytes,
                                       moe_stream_t stream) {
  (void)ws_bytes;
  const moe_dims& d = layer->d;
  const int has_shared = (d.flags & MOE_HAS_SHARED) ? 1 : 0;
  const int has_gate = (d.flags & MOE_HAS_SHARED_GATE) ? 1 : 0;
  const WsLayout L = ws_layout(d, B);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  WsHeader* hdr = at<WsHeader>(ws, 0);
  const int shared_bits = has_shared ? layer->shared_bits : d.bits;
  cudaError_t e;
  if (tc_refused(d, B)) return MOE_ERR_UNSUPPORTED;
  const bool use_tc = B > 1 && (d.flags & MOE_TENSOR_CORES);

  DecodeArgs f;
  if (B == 1 && decode_args_for(d, shared_bits, h, ws, L, &f)) {
    f.ly = decode_layer_of(*layer, logit_offset, idx_out, w_out);
    e = launch_decode(f, (d.flags & MOE_PDL) != 0, s);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e);
  }

  // multi-kernel path (its kernels chained by programmatic launch with MOE_PDL)
  PdlScope pdl_scope((d.flags & MOE_PDL) != 0);
  const int K = d.top_k, E = d.n_experts, H = d.hidden, I = d.inter;
  const int nslots = K + has_shared;
  NormQuantArgs nq{};
  nq.in = h;
  nq.n = H;
  nq.do_norm = 1;
  nq.eps = d.rms_eps;
  nq.gamma = layer->rms_gamma;
  nq.xn_out = at<float>(ws, L.xn);
  nq.q = at<uint8_t>(ws, L.xq);
  nq.e = at<float2>(ws, L.xe);
  nq.hdr = hdr;
  if ((e = launch_norm_quant(nq, B, s)) != cudaSuccess) return cuda_fail(e);

  RouterArgs r{};
  r.xn = nq.xn_out;
  r.B = B;
  r.H = H;
  r.E = E;
  r.router = layer->router;
  r.gate = has_gate ? layer->shared_gate : nullptr;
  r.stages_per_split = router_stages_per_split(B, H, E);
  r.logits = at<float>(ws, L.logits);
  if ((e = launch_router(r, s)) != cudaSuccess) return cuda_fail(e);

  TopkArgs t{};
  t.logits = r.logits;
  t.offset = logit_offset;
  t.B = B;
  t.splits = router_splits(B, H, E);
  t.E = E;
  t.K = K;
  t.has_gate = has_gate;
  t.idx = at<int32_t>(ws, L.idx);
  t.w = at<float>(ws, L.w);
  t.gs = at<float>(ws, L.gs);
  t.idx_out = idx_out;
  t.w_out = w_out;
  t.hdr = hdr;
  if ((e = launch_topk(t, B, s)) != cudaSuccess) return cuda_fail(e);

  BucketArgs bk{};
  bk.idx = t.idx;
  bk.B = B;
  bk.K = K;
  bk.E = E;
  bk.has_shared = has_shared;
  bk.nslots = nslots;
  bk.n_uniq = at<int>(ws, L.nuniq);
  bk.uniq_e = at<int>(ws, L.uniq_e);
  bk.uniq_off = at<int>(ws, L.uniq_off);
  bk.ent = at<int>(ws, L.ent);
  if ((e = launch_bucket(bk, s)) != cudaSuccess) return cuda_fail(e);
  const int items = std::min(B * K, E) + (has_shared ? (B + kSharedChunk - 1) / kSharedChunk : 0);

  if (use_tc) {
    TcSource src{};
    src.experts = static_cast<const uint8_t*>(layer->experts);
    src.stride = layer->expert_stride;
    src.E = E;
    src.bits = d.bits;
    src.shared = static_cast<const uint8_t*>(layer->shared);
    src.shared_bits = shared_bits;
    src.has_shared = has_shared;
    src.xn = nq.xn_out;
    const moe_status st = run_tc(d, L, ws, B, nslots, src, bk.n_uniq, bk.uniq_e, bk.uniq_off, bk.ent, s);
    if (st != MOE_OK) return st;
  } else {
    GateUpArgs g{};
    g.H = H;
    g.I = I;
    g.K = K;
    g.B = B;
    g.nslots = nslots;
    g.bits = d.bits;
    g.shared_bits = shared_bits;
    g.experts = static_cast<const uint8_t*>(layer->experts);
    g.stride = layer->expert_stride;
    g.shared = static_cast<const uint8_t*>(layer->shared);
    g.n_uniq = bk.n_uniq;
    g.uniq_e = bk.uniq_e;
    g.uniq_off = bk.uniq_off;
    g.ent = bk.ent;
    g.xq = nq.q;
    g.xe = nq.e;
    g.a_out = at<float>(ws, L.a);
    if ((e = launch_gateup(g, items, s)) != cudaSuccess) return cuda_fail(e);

    NormQuantArgs aq{};
    aq.in = g.a_out;
    aq.n = I;
    aq.do_norm = 0;
    aq.q = at<uint8_t>(ws, L.aq);
    aq.e = at<float2>(ws, L.ae);
    aq.hdr = hdr;
    if ((e = launch_norm_quant(aq, B * nslots, s)) != cudaSuccess) return cuda_fail(e);

    DownArgs dn{};
    dn.H = H;
    dn.I = I;
    dn.K = K;
    dn.B = B;
    dn.nslots = nslots;
    dn.bits = d.bits;
    dn.shared_bits = shared_bits;
    dn.experts = g.experts;
    dn.stride = g.stride;
    dn.shared = g.shared;
    dn.n_uniq = bk.n_uniq;
    dn.uniq_e = bk.uniq_e;
    dn.uniq_off = bk.uniq_off;
    dn.ent = bk.ent;
    dn.aq = aq.q;
    dn.ae = aq.e;
    dn.d_out = at<float>(ws, L.d);
    if ((e = launch_down(dn, items, s)) != cudaSuccess) return cuda_fail(e);
  }

  CombineArgs cb{};
  cb.B = B;
  cb.H = H;
  cb.K = K;
  cb.nslots = nslots;
  cb.has_shared = has_shared;
  cb.single = 0;
  cb.d = at<float>(ws, L.d);
  cb.w = t.w;
  cb.gs = t.gs;
  cb.out = h;
  if ((e = launch_combine(cb, s)) != cudaSuccess) return cuda_fail(e);
  return MOE_OK;
}

moe_status moe_get_device_status(void* ws, moe_stream_t stream) {
  if (!ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e);
  WsHeader hh;
  e = cudaMemcpy(&hh, ws, sizeof(hh), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (hh.status || hh.abort || hh.bar_extra) {
    // the error state only: the launch counter keeps counting, so that words
    // published before the error can never match a later launch's epoch
    e = cudaMemset(ws, 0, kHeaderErrorBytes);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (hh.status & ST_TIMEOUT) return MOE_ERR_TIMEOUT;
  if (hh.status & ST_NONFINITE) return MOE_ERR_NONFINITE;
  if (hh.status & (tc::ST_RANGE | tc::ST_PLAN | tc::ST_BOUNDS)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_NONFINITE: return "non-finite activation";
  }
  return "unknown status";
}

const char* moe_last_error_message(void) { return g_last_error.c_str(); }

}  // extern "C"
