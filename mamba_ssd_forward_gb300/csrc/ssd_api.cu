// C ABI of libssd_gb300: argument validation, workspace layout and the
// launch sequence.  Every computation happens in the kernels; this file only
// checks arguments and enqueues launches on the caller's stream.
#include <cstdint>
#include <vector>

#include "fwd.cuh"
#include "ssd_internal.cuh"

namespace {

using ssd::Dims;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks shared by every entry point.  INVALID_ARG for malformed
// shapes, UNSUPPORTED for well-formed shapes outside the supported range.
ssd_status check_dims(const ssd_dims *in, Dims *out) {
  if (!in) return SSD_ERR_INVALID_ARG;
  const ssd_dims d = *in;
  if (d.batch < 1 || d.seqlen < 1 || d.nheads < 1 || d.headdim < 1 || d.dstate < 1 ||
      d.ngroups < 1 || d.chunk < 1)
    return SSD_ERR_INVALID_ARG;
  if (d.nheads % d.ngroups != 0) return SSD_ERR_INVALID_ARG;
  if (d.headdim % 16 || d.headdim > 128 || d.dstate % 16 || d.dstate > 256)
    return SSD_ERR_UNSUPPORTED;
  if (d.chunk != 64 && d.chunk != 128 && d.chunk != 256) return SSD_ERR_UNSUPPORTED;
  // Grid limits (batch and heads index grid dimensions) and 62-bit element
  // counts for every tensor.
  if (d.batch > 65535 || d.nheads > 32767 || d.seqlen > 0x7fffffffLL) return SSD_ERR_UNSUPPORTED;
  const int64_t nc = (d.seqlen + d.chunk - 1) / d.chunk;
  const double big = 4.0e18;
  if ((double)d.batch * d.seqlen * d.nheads * d.headdim > big ||
      (double)d.batch * d.nheads * nc * d.headdim * d.dstate > big ||
      (double)d.batch * d.seqlen * d.ngroups * d.dstate > big || nc > (int64_t)1 << 31)
    return SSD_ERR_UNSUPPORTED;
  out->b = d.batch;
  out->L = d.seqlen;
  out->nh = d.nheads;
  out->P = d.headdim;
  out->S = d.dstate;
  out->ng = d.ngroups;
  out->T = d.chunk;
  out->nc = nc;
  out->hpg = d.nheads / d.ngroups;
  return SSD_OK;
}

bool valid_dtype(ssd_dtype t) { return t == SSD_F32 || t == SSD_BF16; }

// Required pointer: non-null and 16-byte aligned.
bool req(const void *p) { return p && aligned16(p); }
// Optional pointer: null, or 16-byte aligned.
bool opt(const void *p) { return !p || aligned16(p); }

ssd_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA; }

// Workspace of ssd_forward: the header (the call's error word), then for
// bf16 I/O the per-chunk start states in bf16, [b, nh, nc, S, P], the chunk
// jump terms, the per-chunk decays, and the factored-decay inputs of the
// fwd_out output kernel (per-token u and v, fp32 [b, nh, nc * T], and the
// per-chunk anchors, float2 [b, nh, nc]); for fp32 I/O G, the chunk jump
// terms and the per-chunk states (fp32, the step-wise layouts).  Each part
// is 256-byte aligned.
struct WsLayout {
  size_t G, dstates, states, u, v, anchor, total;
};

size_t round256(size_t n) { return (n + 255) & ~size_t(255); }

WsLayout ws_layout(const Dims &d, ssd_dtype t) {
  WsLayout w;
  const size_t h = ssd::kWsHeader;
  if (t == SSD_BF16) {
    // header | states (bf16) | jump terms (bf16) | per-chunk (decay, state scale) (fp32 pairs)
    const size_t st = round256(2 * (size_t)(d.b * d.nh * d.nc * d.S * d.P));
    w.states = h;
    w.dstates = h + st;
    w.G = h + 2 * st;
    const size_t tok = round256(sizeof(float) * d.b * d.nh * d.nc * d.T);
    w.u = w.G + round256(2 * sizeof(float) * d.b * d.nh * d.nc);
    w.v = w.u + tok;
    w.anchor = w.v + tok;
    w.total = w.anchor + round256(2 * sizeof(float) * d.b * d.nh * d.nc);
    return w;
  }
  w.G = h;
  w.dstates = h + round256(sizeof(float) * d.b * d.nh * d.nc * d.T);
  const size_t st = round256(sizeof(float) * d.b * d.nh * d.nc * d.P * d.S);
  w.states = w.dstates + st;
  w.u = w.v = w.anchor = 0;
  w.total = w.states + st;
  return w;
}

size_t io_size(ssd_dtype t) { return t == SSD_BF16 ? 2 : 4; }

// The bf16 intermediates of one forward pass, carved from its workspace.
struct Bf16Ws {
  void *states, *dH;
  float2 *gamma;
  float *u, *v;
  float2 *anchor;
};
Bf16Ws bf16_ws(const WsLayout &w, void *workspace) {
  char *ws = static_cast<char *>(workspace);
  Bf16Ws r;
  r.states = ws + w.states;
  r.dH = ws + w.dstates;
  r.gamma = reinterpret_cast<float2 *>(ws + w.G);
  r.u = reinterpret_cast<float *>(ws + w.u);
  r.v = reinterpret_cast<float *>(ws + w.v);
  r.anchor = reinterpret_cast<float2 *>(ws + w.anchor);
  return r;
}

cudaError_t launch_scan(const Dims &d, const ssd::FwdPlan &plan, const void *x, const void *B,
                        const void *C, const void *dt, const float *A, const Bf16Ws &b,
                        const float *D, void *y, int *err, cudaStream_t st) {
  const void *states = b.states;
  if (plan.scan_kernel == 3)
    return ssd::launch_fwd_out(d, x, B, C, dt, A, states, D, b.u, b.v, b.anchor, y,
                               plan.scan_heads, err, st);
  return plan.scan_kernel
             ? ssd::launch_fwd_scan_chunk(d, x, B, C, dt, A, states, D, y, plan.scan_heads,
                                          plan.scan_kernel == 2, err, st)
             : ssd::launch_fwd_scan(d, x, B, C, dt, A, states, D, y, plan.scan_heads, err, st);
}

ssd_plan to_public(const ssd::FwdPlan &p) {
  ssd_plan o;
  o.chunk_state_heads = p.cs.H;
  o.chunk_state_ctas = p.cs.ctas;
  o.scan_kernel = p.scan_kernel;
  o.scan_heads = p.scan_heads;
  return o;
}
ssd::FwdPlan from_public(const ssd_plan &p) {
  ssd::FwdPlan o;
  o.cs = ssd::CsPlan{p.chunk_state_heads, p.chunk_state_ctas};
  o.scan_kernel = p.scan_kernel;
  o.scan_heads = p.scan_heads;
  return o;
}

// The plan a forward call runs: *plan when given (bf16 only, and one of the
// candidates), else the cost-model default.  INVALID_ARG for a plan that is
// not a candidate, or any plan with fp32 I/O.
ssd_status resolve_plan(const Dims &d, ssd_dtype t, const ssd_plan *plan, ssd::FwdPlan *out) {
  if (!plan) {
    if (t == SSD_BF16) *out = ssd::fwd_default_plan(d);
    return SSD_OK;
  }
  if (t != SSD_BF16) return SSD_ERR_INVALID_ARG;
  const ssd::FwdPlan p = from_public(*plan);
  if (!ssd::fwd_plan_ok(d, p)) return SSD_ERR_INVALID_ARG;
  *out = p;
  return SSD_OK;
}

// Mean milliseconds per launch of `launch` over reps launches (after one
// untimed launch), timed with events on st: back to back between two events
// (flush null), or each launch alone after overwriting the flush buffer and
// running `prologue`.
template <typename F, typename Pre>
cudaError_t time_launches(F launch, int reps, cudaStream_t st, cudaEvent_t e0, cudaEvent_t e1,
                          void *flush, size_t flush_bytes, Pre prologue, float *ms) {
  cudaError_t e = launch();
  if (!flush) {
    // back to back: one pair of events around all repetitions
    if (e == cudaSuccess) e = cudaEventRecord(e0, st);
    for (int i = 0; i < reps && e == cudaSuccess; ++i) e = launch();
    if (e == cudaSuccess) e = cudaEventRecord(e1, st);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    if (e == cudaSuccess) e = cudaEventElapsedTime(ms, e0, e1);
    if (e == cudaSuccess) *ms /= (float)reps;
    return e;
  }
  // each repetition after writing the flush buffer and running the
  // prologue (the kernels that precede this one in a forward pass), both
  // outside the events, so every launch sees the cache state it would see
  // in a forward pass over fresh inputs
  float total = 0.f;
  for (int i = 0; i < reps && e == cudaSuccess; ++i) {
    e = cudaMemsetAsync(flush, i & 0xff, flush_bytes, st);
    if (e == cudaSuccess) e = prologue();
    if (e == cudaSuccess) e = cudaEventRecord(e0, st);
    if (e == cudaSuccess) e = launch();
    if (e == cudaSuccess) e = cudaEventRecord(e1, st);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    float one = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&one, e0, e1);
    total += one;
  }
  if (e == cudaSuccess) *ms = total / (float)reps;
  return e;
}

// Device workspace of ssd_forward_host: the forward's own workspace, then a
// device copy of every input and output, each 256-byte aligned.
struct HostLayout {
  size_t fwd, fwd_bytes, x, dt, A, B, C, D, h0, y, fin, total;
};

HostLayout host_layout(const Dims &d, ssd_dtype t, int has_D, int has_h0, int has_fin) {
  HostLayout h;
  const size_t e = io_size(t);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += round256(bytes);
    return at;
  };
  h.fwd_bytes = ws_layout(d, t).total;
  h.fwd = take(h.fwd_bytes);
  h.x = take(e * d.b * d.L * d.nh * d.P);
  h.dt = take(e * d.b * d.L * d.nh);
  h.A = take(sizeof(float) * d.nh);
  h.B = take(e * d.b * d.L * d.ng * d.S);
  h.C = take(e * d.b * d.L * d.ng * d.S);
  h.D = take(has_D ? sizeof(float) * d.nh : 0);
  h.h0 = take(has_h0 ? sizeof(float) * d.b * d.nh * d.P * d.S : 0);
  h.y = take(e * d.b * d.L * d.nh * d.P);
  h.fin = take(has_fin ? sizeof(float) * d.b * d.nh * d.P * d.S : 0);
  h.total = off;
  return h;
}

}  // namespace

extern "C" {

const char *ssd_status_string(ssd_status s) {
  switch (s) {
    case SSD_OK: return "SSD_OK";
    case SSD_ERR_INVALID_ARG: return "SSD_ERR_INVALID_ARG: null, misaligned or malformed argument";
    case SSD_ERR_UNSUPPORTED: return "SSD_ERR_UNSUPPORTED: dimensions outside the supported range";
    case SSD_ERR_CUDA: return "SSD_ERR_CUDA: a CUDA call or kernel launch failed";
    case SSD_ERR_TIMEOUT: return "SSD_ERR_TIMEOUT: a bounded device-side wait gave up";
    case SSD_ERR_BOUNDS:
      return "SSD_ERR_BOUNDS: a debug-bounds build caught an out-of-range access";
  }
  return "SSD_ERR_UNKNOWN";
}

ssd_status ssd_device_error(void *stream) {
  int *word = ssd::device_error_word();
  int code = 0;
  if (!word || ssd::read_and_clear_error(word, (cudaStream_t)stream, &code) != cudaSuccess)
    return SSD_ERR_CUDA;
  return ssd::status_of_error_code(code);
}

ssd_status ssd_workspace_error(void *workspace, void *stream) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return SSD_ERR_INVALID_ARG;
  int code = 0;
  if (ssd::read_and_clear_error(static_cast<int *>(workspace), (cudaStream_t)stream, &code) !=
      cudaSuccess)
    return SSD_ERR_CUDA;
  return ssd::status_of_error_code(code);
}

size_t ssd_forward_workspace_size(const ssd_dims *dims, ssd_dtype dtype) {
  Dims d;
  if (!valid_dtype(dtype) || check_dims(dims, &d) != SSD_OK) return 0;
  return ws_layout(d, dtype).total;
}

ssd_status ssd_chunk_cumsum(const ssd_dims *dims, ssd_dtype dtype, const void *dt,
                            const float *A, float *G, void *stream) {
  Dims d;
  ssd_status s = check_dims(dims, &d);
  if (s != SSD_OK) return s;
  if (!valid_dtype(dtype) || !req(dt) || !req(A) || !req(G)) return SSD_ERR_INVALID_ARG;
  int *err = ssd::device_error_word();
  if (!err) return SSD_ERR_CUDA;
  return from_cuda(ssd::launch_chunk_cumsum(d, dtype, dt, A, G, err, (cudaStream_t)stream));
}

ssd_status ssd_chunk_state(const ssd_dims *dims, ssd_dtype dtype, const void *x,
                           const void *B, const void *dt, const float *G, float *dstates,
                           void *stream) {
  Dims d;
  ssd_status s = check_dims(dims, &d);
  if (s != SSD_OK) return s;
  if (!valid_dtype(dtype) || !req(x) || !req(B) || !req(dt) || !req(G) || !req(dstates))
    return SSD_ERR_INVALID_ARG;
  int *err = ssd::device_error_word();
  if (!err) return SSD_ERR_CUDA;
  return from_cuda(
      ssd::launch_chunk_state(d, dtype, x, B, dt, G, dstates, err, (cudaStream_t)stream));
}

ssd_status ssd_state_passing(const ssd_dims *dims, const float *dstates, const float *G,
                             const float *h0, float *states, float *final_state,
                             void *stream) {
  Dims d;
  ssd_status s = check_dims(dims, &d);
  if (s != SSD_OK) return s;
  if (!req(dstates) || !req(G) || !opt(h0) || !req(states) || !opt(final_state))
    return SSD_ERR_INVALID_ARG;
  int *err = ssd::device_error_word();
  if (!err) return SSD_ERR_CUDA;
  return from_cuda(ssd::launch_state_passing(d, dstates, G, h0, states, final_state, err,
                                             (cudaStream_t)stream));
}

ssd_status ssd_chunk_scan(const ssd_dims *dims, ssd_dtype dtype, const void *x, const void *B,
                          const void *C, const void *dt, const float *G, const float *states,
                          const float *D, void *y, void *stream) {
  Dims d;
  ssd_status s = check_dims(dims, &d);
  if (s != SSD_OK) return s;
  if (!valid_dtype(dtype) || !req(x) || !req(B) || !req(C) || !req(dt) || !req(G) ||
      !req(states) || !opt(D) || !req(y))
    return SSD_ERR_INVALID_ARG;
  int *err = ssd::device_error_word();
  if (!err) return SSD_ERR_CUDA;
  return from_cuda(ssd::launch_chunk_scan(d, dtype, x, B, C, dt, G, states, D, y, err,
                                          (cudaStream_t)stream));
}

ssd_status ssd_decode_step(const ssd_dims *dims, ssd_dtype dtype, const void *x, const void *dt,
                           const float *A, const void *B, const void *C, const float *D,
                           float *state, void *y, void *stream) {
  if (!dims) return SSD_ERR_INVALID_ARG;
  const ssd_dims d = *dims;
  if (d.batch < 1 || d.nheads < 1 || d.headdim < 1 || d.dstate < 1 || d.ngroups < 1 ||
      d.seqlen != 1 || d.nheads % d.ngroups != 0)
    return SSD_ERR_INVALID_ARG;
  if (d.dstate % 4 || d.dstate > 1024 || d.headdim > (1 << 20) ||
      (double)d.batch * d.nheads > 2147483647.0 ||
      (double)d.batch * d.nheads * d.headdim * d.dstate > 4.0e18)
    return SSD_ERR_UNSUPPORTED;
  if (!valid_dtype(dtype) || !req(x) || !req(dt) || !req(A) || !req(B) || !req(C) || !opt(D) ||
      !req(state) || !req(y))
    return SSD_ERR_INVALID_ARG;
  int *err = ssd::device_error_word();
  if (!err) return SSD_ERR_CUDA;
  return from_cuda(ssd::launch_decode_step(d.batch, d.nheads, d.headdim, d.dstate, d.ngroups,
                                           dtype, x, dt, A, B, C, D, state, y, err,
                                           (cudaStream_t)stream));
}

}  // extern "C"

namespace ssd {

ssd_status check_forward_args(const ssd_dims *dims, ssd_dtype dtype, const void *x,
                              const void *dt, const float *A, const void *B, const void *C,
                              const float *D, const float *h0, const void *y,
                              const float *final_state, Dims *out) {
  ssd_status s = check_dims(dims, out);
  if (s != SSD_OK) return s;
  if (!valid_dtype(dtype) || !req(x) || !req(dt) || !req(A) || !req(B) || !req(C) ||
      !opt(D) || !opt(h0) || !req(y) || !opt(final_state))
    return SSD_ERR_INVALID_ARG;
  return SSD_OK;
}

ssd_status plan_status(const ssd_dims *dims, ssd_dtype dtype, const ssd_plan *plan) {
  Dims d;
  const ssd_status s = check_dims(dims, &d);
  if (s != SSD_OK) return s;
  if (!valid_dtype(dtype)) return SSD_ERR_INVALID_ARG;
  ssd::FwdPlan fp{};
  return resolve_plan(d, dtype, plan, &fp);
}

ssd_status forward_impl(const ssd_dims *dims, ssd_dtype dtype, const void *x, const void *dt,
                        const float *A, const void *B, const void *C, const float *D,
                        const float *h0, void *y, float *final_state, void *workspace,
                        size_t ws_bytes, const ssd_plan *plan, int *err, cudaStream_t st,
                        void *const *events, int n_events, int *n_launches) {
  Dims d;
  ssd_status s = check_forward_args(dims, dtype, x, dt, A, B, C, D, h0, y, final_state, &d);
  if (s != SSD_OK) return s;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || n_events < 0 ||
      (n_events > 0 && !events))
    return SSD_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(d, dtype);
  if (ws_bytes < w.total) return SSD_ERR_INVALID_ARG;
  ssd::FwdPlan fp{};
  s = resolve_plan(d, dtype, plan, &fp);
  if (s != SSD_OK) return s;
  if (!err) err = static_cast<int *>(workspace);  // the workspace's own error word
  char *ws = static_cast<char *>(workspace);
  int launched = 0;
  auto mark = [&](int i) -> cudaError_t {
    if (events && i < n_events) return cudaEventRecord((cudaEvent_t)events[i], st);
    return cudaSuccess;
  };
  cudaError_t e = mark(0);
  if (dtype == SSD_BF16) {
    // chunk jump terms (all chunks in parallel), the sequential pass over
    // chunks, then the output pass; with the factored output kernel the
    // first also writes its per-token factors and anchors and the second
    // stores the start states scaled by them
    const Bf16Ws bw = bf16_ws(w, workspace);
    const bool fac = fp.scan_kernel == 3;
    if (e == cudaSuccess)
      e = ssd::launch_fwd_chunk_state(d, x, B, dt, A, bw.dH, bw.gamma, fac ? bw.u : nullptr,
                                      fac ? bw.v : nullptr, fac ? bw.anchor : nullptr, fp.cs,
                                      err, st);
    if (e == cudaSuccess && ++launched) e = mark(launched);
    if (e == cudaSuccess)
      e = ssd::launch_fwd_state_pass(d, bw.dH, bw.gamma, h0, bw.states, final_state, err, st);
    if (e == cudaSuccess && ++launched) e = mark(launched);
    if (e == cudaSuccess) e = launch_scan(d, fp, x, B, C, dt, A, bw, D, y, err, st);
    if (e == cudaSuccess && ++launched) e = mark(launched);
  } else {
    float *G = reinterpret_cast<float *>(ws + w.G);
    float *dst = reinterpret_cast<float *>(ws + w.dstates);
    float *sts = reinterpret_cast<float *>(ws + w.states);
    // the cumsum and the chunk jump terms: the warp-specialised tf32 kernel,
    // which forms G itself, where the shape allows; else the two step kernels
    if (ssd::fwd_chunk_state_tf32_supported(d)) {
      if (e == cudaSuccess)
        e = ssd::launch_fwd_chunk_state_tf32(d, static_cast<const float *>(x),
                                             static_cast<const float *>(B),
                                             static_cast<const float *>(dt), A, G, dst, err, st);
    } else {
      if (e == cudaSuccess) e = ssd::launch_chunk_cumsum(d, dtype, dt, A, G, err, st);
      if (e == cudaSuccess && ++launched) e = mark(launched);
      if (e == cudaSuccess) e = ssd::launch_chunk_state(d, dtype, x, B, dt, G, dst, err, st);
    }
    if (e == cudaSuccess && ++launched) e = mark(launched);
    // the output pass: the warp-specialised tf32 kernel where the shape
    // allows (it reads the stored states rounded to tf32), else the step
    // kernel
    const bool fast = ssd::fwd_out_tf32_supported(d);
    if (e == cudaSuccess)
      e = ssd::launch_state_passing(d, dst, G, h0, sts, final_state, err, st, fast);
    if (e == cudaSuccess && ++launched) e = mark(launched);
    if (e == cudaSuccess)
      e = fast ? ssd::launch_fwd_out_tf32(d, static_cast<const float *>(x),
                                          static_cast<const float *>(B),
                                          static_cast<const float *>(C),
                                          static_cast<const float *>(dt), G, sts, D,
                                          static_cast<float *>(y), ssd::fwd_out_tf32_heads(d),
                                          err, st)
               : ssd::launch_chunk_scan(d, dtype, x, B, C, dt, G, sts, D, y, err, st);
    if (e == cudaSuccess && ++launched) e = mark(launched);
  }
  if (n_launches) *n_launches = launched;
  return from_cuda(e);
}

}  // namespace ssd

extern "C" {

ssd_status ssd_forward(const ssd_dims *dims, ssd_dtype dtype, const void *x, const void *dt,
                       const float *A, const void *B, const void *C, const float *D,
                       const float *h0, void *y, float *final_state, void *workspace,
                       size_t ws_bytes, void *stream) {
  return ssd::forward_impl(dims, dtype, x, dt, A, B, C, D, h0, y, final_state, workspace,
                           ws_bytes, nullptr, nullptr, (cudaStream_t)stream, nullptr, 0, nullptr);
}

ssd_status ssd_forward_ex(const ssd_dims *dims, ssd_dtype dtype, const void *x, const void *dt,
                          const float *A, const void *B, const void *C, const float *D,
                          const float *h0, void *y, float *final_state, void *workspace,
                          size_t ws_bytes, const ssd_plan *plan, void *stream) {
  return ssd::forward_impl(dims, dtype, x, dt, A, B, C, D, h0, y, final_state, workspace,
                           ws_bytes, plan, nullptr, (cudaStream_t)stream, nullptr, 0, nullptr);
}

ssd_status ssd_forward_profiled(const ssd_dims *dims, ssd_dtype dtype, const void *x,
                                const void *dt, const float *A, const void *B, const void *C,
                                const float *D, const float *h0, void *y, float *final_state,
                                void *workspace, size_t ws_bytes, const ssd_plan *plan,
                                void *stream, void *const *events, int n_events,
                                int *n_launches) {
  return ssd::forward_impl(dims, dtype, x, dt, A, B, C, D, h0, y, final_state, workspace,
                           ws_bytes, plan, nullptr, (cudaStream_t)stream, events, n_events,
                           n_launches);
}

int ssd_forward_plan_candidates(const ssd_dims *dims, ssd_dtype dtype, ssd_plan *out,
                                int max_out) {
  Dims d;
  if (dtype != SSD_BF16 || check_dims(dims, &d) != SSD_OK || max_out < 0 ||
      (max_out > 0 && !out))
    return 0;
  std::vector<ssd::CsPlan> cs;
  std::vector<ssd::FwdPlan> sc;
  ssd::fwd_cs_candidates(d, &cs);
  ssd::fwd_scan_candidates(d, &sc);
  int n = 0;
  for (const ssd::CsPlan &c : cs)
    for (ssd::FwdPlan p : sc) {
      p.cs = c;
      if (n < max_out) out[n] = to_public(p);
      ++n;
    }
  return n;
}

ssd_status ssd_forward_default_plan(const ssd_dims *dims, ssd_dtype dtype, ssd_plan *out) {
  Dims d;
  const ssd_status s = check_dims(dims, &d);
  if (s != SSD_OK) return s;
  if (!valid_dtype(dtype) || !out) return SSD_ERR_INVALID_ARG;
  if (dtype != SSD_BF16) return SSD_ERR_UNSUPPORTED;
  *out = to_public(ssd::fwd_default_plan(d));
  return SSD_OK;
}

ssd_status ssd_forward_tune(const ssd_dims *dims, ssd_dtype dtype, const void *x, const void *dt,
                            const float *A, const void *B, const void *C, const float *D,
                            const float *h0, void *y, float *final_state, void *workspace,
                            size_t ws_bytes, int reps, void *flush, size_t flush_bytes,
                            void *stream, ssd_plan *chosen) {
  Dims d;
  ssd_status s = ssd::check_forward_args(dims, dtype, x, dt, A, B, C, D, h0, y, final_state, &d);
  if (s != SSD_OK) return s;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || reps < 1 ||
      reps > 1000 || !chosen || (flush && flush_bytes == 0))
    return SSD_ERR_INVALID_ARG;
  if (dtype != SSD_BF16) return SSD_ERR_UNSUPPORTED;
  const WsLayout w = ws_layout(d, dtype);
  if (ws_bytes < w.total) return SSD_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  int *err = static_cast<int *>(workspace);
  // the start states the output kernels read, from one pass with the
  // default plan
  s = ssd_forward(dims, dtype, x, dt, A, B, C, D, h0, y, final_state, workspace, ws_bytes,
                  stream);
  if (s != SSD_OK) return s;
  const Bf16Ws bw = bf16_ws(w, workspace);
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  cudaError_t e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  ssd::FwdPlan best = ssd::fwd_default_plan(d);
  std::vector<ssd::CsPlan> cs;
  std::vector<ssd::FwdPlan> sc;
  ssd::fwd_cs_candidates(d, &cs);
  ssd::fwd_scan_candidates(d, &sc);
  float best_ms = 3.0e38f;
  for (size_t i = 0; i < cs.size() && e == cudaSuccess; ++i) {
    float ms = 0.f;
    e = time_launches(
        [&] {
          return ssd::launch_fwd_chunk_state(d, x, B, dt, A, bw.dH, bw.gamma, bw.u, bw.v,
                                             bw.anchor, cs[i], err, st);
        },
        reps, st, e0, e1, flush, flush_bytes, [] { return cudaSuccess; }, &ms);
    if (e == cudaSuccess && ms < best_ms) {
      best_ms = ms;
      best.cs = cs[i];
    }
  }
  best_ms = 3.0e38f;
  for (size_t i = 0; i < sc.size() && e == cudaSuccess; ++i) {
    float ms = 0.f;
    // with a flush buffer each output launch follows the chunk-jump kernel
    // (the plan chosen above) and the state pass, as in a forward pass
    e = time_launches(
        [&] { return launch_scan(d, sc[i], x, B, C, dt, A, bw, D, y, err, st); }, reps, st, e0,
        e1, flush, flush_bytes,
        [&] {
          cudaError_t e2 = ssd::launch_fwd_chunk_state(d, x, B, dt, A, bw.dH, bw.gamma, bw.u,
                                                       bw.v, bw.anchor, best.cs, err, st);
          if (e2 == cudaSuccess)
            e2 = ssd::launch_fwd_state_pass(d, bw.dH, bw.gamma, h0, bw.states, final_state, err,
                                            st);
          return e2;
        },
        &ms);
    if (e == cudaSuccess && ms < best_ms) {
      best_ms = ms;
      best.scan_kernel = sc[i].scan_kernel;
      best.scan_heads = sc[i].scan_heads;
    }
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (e != cudaSuccess) return SSD_ERR_CUDA;
  const ssd_plan pub = to_public(best);
  s = ssd_forward_ex(dims, dtype, x, dt, A, B, C, D, h0, y, final_state, workspace, ws_bytes,
                     &pub, stream);
  if (s != SSD_OK) return s;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SSD_ERR_CUDA;
  *chosen = pub;
  return SSD_OK;
}

size_t ssd_forward_host_workspace_size(const ssd_dims *dims, ssd_dtype dtype, int has_D,
                                       int has_h0, int want_final_state) {
  Dims d;
  if (!valid_dtype(dtype) || check_dims(dims, &d) != SSD_OK) return 0;
  return host_layout(d, dtype, has_D, has_h0, want_final_state).total;
}

ssd_status ssd_forward_host(const ssd_dims *dims, ssd_dtype dtype, const void *x,
                            const void *dt, const float *A, const void *B, const void *C,
                            const float *D, const float *h0, void *y, float *final_state,
                            void *workspace, size_t ws_bytes, const ssd_plan *plan,
                            void *stream) {
  Dims d;
  ssd_status s = check_dims(dims, &d);
  if (s != SSD_OK) return s;
  if (!valid_dtype(dtype) || !x || !dt || !A || !B || !C || !y || !workspace ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return SSD_ERR_INVALID_ARG;
  ssd::FwdPlan fp{};
  s = resolve_plan(d, dtype, plan, &fp);
  if (s != SSD_OK) return s;
  const HostLayout hl = host_layout(d, dtype, D != nullptr, h0 != nullptr, final_state != nullptr);
  if (ws_bytes < hl.total) return SSD_ERR_INVALID_ARG;
  char *ws = static_cast<char *>(workspace);
  cudaStream_t st = (cudaStream_t)stream;
  const size_t e = io_size(dtype);
  cudaError_t err = cudaSuccess;
  auto h2d = [&](size_t off, const void *src, size_t bytes) {
    if (err == cudaSuccess && src)
      err = cudaMemcpyAsync(ws + off, src, bytes, cudaMemcpyHostToDevice, st);
  };
  h2d(hl.x, x, e * d.b * d.L * d.nh * d.P);
  h2d(hl.dt, dt, e * d.b * d.L * d.nh);
  h2d(hl.A, A, sizeof(float) * d.nh);
  h2d(hl.B, B, e * d.b * d.L * d.ng * d.S);
  h2d(hl.C, C, e * d.b * d.L * d.ng * d.S);
  h2d(hl.D, D, sizeof(float) * d.nh);
  h2d(hl.h0, h0, sizeof(float) * d.b * d.nh * d.P * d.S);
  if (err != cudaSuccess) return SSD_ERR_CUDA;
  // the forward's workspace sits at offset 0, so its error word is this
  // workspace's
  s = ssd_forward_ex(dims, dtype, ws + hl.x, ws + hl.dt, reinterpret_cast<float *>(ws + hl.A),
                     ws + hl.B, ws + hl.C, D ? reinterpret_cast<float *>(ws + hl.D) : nullptr,
                     h0 ? reinterpret_cast<float *>(ws + hl.h0) : nullptr, ws + hl.y,
                     final_state ? reinterpret_cast<float *>(ws + hl.fin) : nullptr,
                     ws + hl.fwd, hl.fwd_bytes, plan, stream);
  if (s != SSD_OK) return s;
  err = cudaMemcpyAsync(y, ws + hl.y, e * d.b * d.L * d.nh * d.P, cudaMemcpyDeviceToHost, st);
  if (err == cudaSuccess && final_state)
    err = cudaMemcpyAsync(final_state, ws + hl.fin, sizeof(float) * d.b * d.nh * d.P * d.S,
                          cudaMemcpyDeviceToHost, st);
  return from_cuda(err);
}

}  // extern "C"

namespace {

// Workspace of ssd_backward (fp32): the header (the call's error word), G,
// the chunk jump terms (the forward's, then the adjoint's), the start states
// h_k and the adjoint states R_k (both chunk-major), the forward's final
// state, the per-token q . B, dL/dG and gy . x, the per-chunk shares of dA
// and dD, c_i . B_j of every chunk and group (T x T), the head slices' dB,
// dC shares (when a group's heads are split), the state terms dxS, ysmS and
// the scaled inputs x~, gy~ (in the layout of x); with bf16 I/O then fp32
// copies of x, dt, B, C, gy and fp32 buffers for dx, ddt, dB, dC.  Each part
// is 256-byte aligned.
struct BwdLayout {
  size_t G, dst, states, R, fin, qB, dG, gyx, part, Kcb, sB, sC, dxS, ysmS, xs, gys;
  size_t cx, cdt, cB, cC, cgy, cdx, cddt, cdB, cdC;  // bf16 I/O only
  size_t total;
};

BwdLayout bwd_layout(const Dims &d, ssd_dtype dtype) {
  BwdLayout w{};
  const size_t tok = round256(sizeof(float) * d.b * d.nh * d.nc * d.T);
  const size_t st = round256(sizeof(float) * d.b * d.nh * d.nc * d.P * d.S);
  w.G = ssd::kWsHeader;
  w.dst = w.G + tok;
  w.states = w.dst + st;
  w.R = w.states + st;
  w.fin = w.R + st;
  w.qB = w.fin + round256(sizeof(float) * d.b * d.nh * d.P * d.S);
  w.dG = w.qB + tok;
  w.gyx = w.dG + tok;
  w.part = w.gyx + tok;
  w.Kcb = w.part + round256(2 * sizeof(float) * d.b * d.nh * d.nc);
  w.sB = w.Kcb + round256(sizeof(float) * d.b * d.ng * d.nc * d.T * d.T);
  // the head slices' shares of dB and dC, when a group's heads are split
  const int ns = ssd::bwd_head_slices(d);
  const size_t slc = ns > 1 ? round256(sizeof(float) * ns * d.b * d.L * d.ng * d.S) : 0;
  w.sC = w.sB + slc;
  // the state terms' GEMMs: their results dxS, ysmS and scaled inputs x~,
  // gy~ (each in the layout of x)
  const size_t xsz = round256(sizeof(float) * d.b * d.L * d.nh * d.P);
  w.dxS = w.sC + slc;
  w.ysmS = w.dxS + xsz;
  w.xs = w.ysmS + xsz;
  w.gys = w.xs + xsz;
  w.total = w.gys + xsz;
  if (dtype == SSD_BF16) {
    const size_t xs = round256(sizeof(float) * d.b * d.L * d.nh * d.P),
                 ts = round256(sizeof(float) * d.b * d.L * d.nh),
                 gs = round256(sizeof(float) * d.b * d.L * d.ng * d.S);
    w.cx = w.total;
    w.cdt = w.cx + xs;
    w.cB = w.cdt + ts;
    w.cC = w.cB + gs;
    w.cgy = w.cC + gs;
    w.cdx = w.cgy + xs;
    w.cddt = w.cdx + xs;
    w.cdB = w.cddt + ts;
    w.cdC = w.cdB + gs;
    w.total = w.cdC + gs;
  }
  return w;
}

ssd_status check_backward_dims(const ssd_dims *dims, ssd_dtype dtype, Dims *d) {
  const ssd_status s = check_dims(dims, d);
  if (s != SSD_OK) return s;
  if (!valid_dtype(dtype)) return SSD_ERR_INVALID_ARG;
  if (!ssd::bwd_supported(*d)) return SSD_ERR_UNSUPPORTED;
  return SSD_OK;
}

// ssd_backward and ssd_backward_profiled: events (n_events of them, may be
// none) are recorded before the first launch and after each launch.
ssd_status backward_impl(const ssd_dims *dims, ssd_dtype dtype, const void *x, const void *dt,
                         const float *A, const void *B, const void *C, const float *D,
                         const float *h0, const void *gy, const float *gfinal, void *dx,
                         void *ddt, float *dA, void *dB, void *dC, float *dD, float *dh0,
                         void *workspace, size_t ws_bytes, cudaStream_t st,
                         void *const *events, int n_events, int *n_launches) {
  Dims d;
  ssd_status s = check_backward_dims(dims, dtype, &d);
  if (s != SSD_OK) return s;
  if (!req(x) || !req(dt) || !req(A) || !req(B) || !req(C) || !opt(D) || !opt(h0) ||
      !req(gy) || !opt(gfinal) || !req(dx) || !req(ddt) || !req(dA) || !req(dB) || !req(dC) ||
      !opt(dD) || !opt(dh0) || !workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
      n_events < 0 || (n_events > 0 && !events))
    return SSD_ERR_INVALID_ARG;
  const BwdLayout w = bwd_layout(d, dtype);
  if (ws_bytes < w.total) return SSD_ERR_INVALID_ARG;
  int *err = static_cast<int *>(workspace);
  char *ws = static_cast<char *>(workspace);
  auto f = [&](size_t off) { return reinterpret_cast<float *>(ws + off); };
  // bf16 I/O: the fp32 pass below reads fp32 copies of the inputs and writes
  // fp32 gradients into the workspace, converted to bf16 at the end
  const bool bf = dtype == SSD_BF16;
  const float *xf = bf ? f(w.cx) : static_cast<const float *>(x),
              *dtf = bf ? f(w.cdt) : static_cast<const float *>(dt),
              *Bf = bf ? f(w.cB) : static_cast<const float *>(B),
              *Cf = bf ? f(w.cC) : static_cast<const float *>(C),
              *gyf = bf ? f(w.cgy) : static_cast<const float *>(gy);
  float *dxf = bf ? f(w.cdx) : static_cast<float *>(dx),
        *ddtf = bf ? f(w.cddt) : static_cast<float *>(ddt),
        *dBf = bf ? f(w.cdB) : static_cast<float *>(dB),
        *dCf = bf ? f(w.cdC) : static_cast<float *>(dC);
  float *G = f(w.G), *dst = f(w.dst), *sts = f(w.states), *R = f(w.R), *fin = f(w.fin);
  const bool sliced = ssd::bwd_head_slices(d) > 1;
  const int64_t n_x = d.b * d.L * d.nh * d.P, n_t = d.b * d.L * d.nh,
                n_g = d.b * d.L * d.ng * d.S;
  int launched = 0;
  auto mark = [&](int i) -> cudaError_t {
    if (events && i < n_events) return cudaEventRecord((cudaEvent_t)events[i], st);
    return cudaSuccess;
  };
  // runs one launch unless an earlier step failed, then records its event
  cudaError_t e = mark(0);
  auto step = [&](auto &&launch) {
    if (e == cudaSuccess) e = launch();
    if (e == cudaSuccess) e = mark(++launched);
  };
  if (bf) {
    ssd::BwdConvert cv{};
    cv.seg[0] = {x, f(w.cx), n_x};
    cv.seg[1] = {dt, f(w.cdt), n_t};
    cv.seg[2] = {B, f(w.cB), n_g};
    cv.seg[3] = {C, f(w.cC), n_g};
    cv.seg[4] = {gy, f(w.cgy), n_x};
    cv.nseg = 5;
    cv.to_bf16 = 0;
    step([&] { return ssd::launch_bwd_convert(cv, st); });
  }
  // the forward's cumsum, the scaled inputs x~ = dt exp2(G_last - G) x and
  // gy~ = exp2(G) gy, the jump terms, start states and final state (the
  // forward's own jump kernels take plain TF32 products)
  step([&] { return ssd::launch_chunk_cumsum(d, SSD_F32, dtf, A, G, err, st); });
  step([&] {
    return ssd::launch_bwd_scale(d, xf, gyf, dtf, G, f(w.xs), f(w.gys), err, st);
  });
  step([&] {
    return ssd::launch_bwd_gemm(d, 2, 1, f(w.xs), nullptr, Bf, nullptr, dst, nullptr, err, st);
  });
  step([&] {
    return ssd::launch_state_passing(d, dst, G, h0, sts, fin, err, st, false, false, true);
  });
  // the adjoint: its jump terms (over the forward's, no longer needed), the
  // backward pass over chunks for R_k and dh0, then the per-token gradients
  step([&] {
    return ssd::launch_bwd_gemm(d, 2, 1, f(w.gys), nullptr, Cf, nullptr, dst, nullptr, err, st);
  });
  step([&] {
    return ssd::launch_state_passing(d, dst, G, gfinal, R, dh0, err, st, false, true, true);
  });
  // Kcb: c_i . B_j per chunk and group
  step([&] {
    return ssd::launch_bwd_gemm(d, 3, 1, Cf, nullptr, Bf, nullptr, f(w.Kcb), nullptr, err, st);
  });
  // the state terms: dxS, ysmS before the per-token kernel, dB and dC after it
  step([&] {
    return ssd::launch_bwd_gemm(d, 0, 2, Bf, Cf, R, sts, f(w.dxS), f(w.ysmS), err, st);
  });
  step([&] {
    return ssd::launch_bwd_main(d, xf, dtf, Bf, Cf, D, gyf, G, f(w.dxS), f(w.ysmS), f(w.Kcb), dxf,
                                sliced ? f(w.sB) : dBf, sliced ? f(w.sC) : dCf, f(w.qB),
                                f(w.dG), f(w.gyx), err, st);
  });
  float2 *part = reinterpret_cast<float2 *>(ws + w.part);
  step([&] {
    return ssd::launch_bwd_finish(d, dtf, A, R, sts, fin, f(w.qB), f(w.dG), f(w.gyx), ddtf, part,
                                  err, st);
  });
  step([&] {
    return ssd::launch_bwd_reduce(d, f(w.sB), f(w.sC), dBf, dCf, part, dA, dD, err, st);
  });
  step([&] {
    return ssd::launch_bwd_gemm(d, 1, 2, f(w.xs), f(w.gys), R, sts, dBf, dCf, err, st);
  });
  if (bf) {
    ssd::BwdConvert cv{};
    cv.seg[0] = {dxf, dx, n_x};
    cv.seg[1] = {ddtf, ddt, n_t};
    cv.seg[2] = {dBf, dB, n_g};
    cv.seg[3] = {dCf, dC, n_g};
    cv.nseg = 4;
    cv.to_bf16 = 1;
    step([&] { return ssd::launch_bwd_convert(cv, st); });
  }
  if (n_launches) *n_launches = launched;
  return from_cuda(e);
}

}  // namespace

extern "C" {

size_t ssd_backward_workspace_size(const ssd_dims *dims, ssd_dtype dtype) {
  Dims d;
  if (check_backward_dims(dims, dtype, &d) != SSD_OK) return 0;
  return bwd_layout(d, dtype).total;
}

ssd_status ssd_backward(const ssd_dims *dims, ssd_dtype dtype, const void *x, const void *dt,
                        const float *A, const void *B, const void *C, const float *D,
                        const float *h0, const void *gy, const float *gfinal, void *dx,
                        void *ddt, float *dA, void *dB, void *dC, float *dD, float *dh0,
                        void *workspace, size_t ws_bytes, void *stream) {
  return backward_impl(dims, dtype, x, dt, A, B, C, D, h0, gy, gfinal, dx, ddt, dA, dB, dC, dD,
                       dh0, workspace, ws_bytes, (cudaStream_t)stream, nullptr, 0, nullptr);
}

ssd_status ssd_backward_profiled(const ssd_dims *dims, ssd_dtype dtype, const void *x,
                                 const void *dt, const float *A, const void *B, const void *C,
                                 const float *D, const float *h0, const void *gy,
                                 const float *gfinal, void *dx, void *ddt, float *dA, void *dB,
                                 void *dC, float *dD, float *dh0, void *workspace,
                                 size_t ws_bytes, void *stream, void *const *events,
                                 int n_events, int *n_launches) {
  return backward_impl(dims, dtype, x, dt, A, B, C, D, h0, gy, gfinal, dx, ddt, dA, dB, dC, dD,
                       dh0, workspace, ws_bytes, (cudaStream_t)stream, events, n_events,
                       n_launches);
}

}  // extern "C"
