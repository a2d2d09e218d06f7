// ssd_forward_host_overlapped: the forward pass on host buffers with the
// host<->device copies overlapped with the computation.  The work is cut
// into slices -- along the batch, or (batch 1) along the tokens with each
// slice starting from the previous slice's final state (the resume property
// of the recurrence) -- and three caller streams carry the uploads, the
// forward passes and the downloads, ordered by events created in the call.
// Slice i+1 uploads while slice i computes and slice i-1 downloads.  Only
// argument marshalling and stream ordering live here; every step of the
// method runs in the kernels behind ssd_forward.
#include <algorithm>
#include <vector>

#include "ssd_internal.cuh"

namespace {

struct Slice {
  int64_t b0, nb, t0, nt;  // batch and token range
};

size_t r256(size_t n) { return (n + 255) & ~size_t(255); }

bool valid_dims(const ssd_dims *dims) {
  return dims && ssd_forward_workspace_size(dims, SSD_BF16) > 0;
}

// Slices of the work: min(n, b) along the batch when b >= 2, else up to n
// runs of whole chunks along the tokens.
std::vector<Slice> plan_slices(const ssd_dims &d, int n) {
  std::vector<Slice> out;
  if (d.batch >= 2) {
    const int64_t k = std::min<int64_t>(n, d.batch);
    for (int64_t i = 0; i < k; ++i) {
      const int64_t b0 = i * d.batch / k, b1 = (i + 1) * d.batch / k;
      out.push_back(Slice{b0, b1 - b0, 0, d.seqlen});
    }
  } else {
    const int64_t nc = (d.seqlen + d.chunk - 1) / d.chunk;
    const int64_t k = std::min<int64_t>(n, nc);
    const int64_t per = (nc + k - 1) / k;  // chunks per slice
    for (int64_t t0 = 0; t0 < d.seqlen; t0 += per * d.chunk)
      out.push_back(Slice{0, 1, t0, std::min(per * d.chunk, d.seqlen - t0)});
  }
  return out;
}

// x, dt and y go through double buffers slice by slice (each slice's dt
// then starts on a 256-byte boundary, as ssd_forward needs 16); B and C have
// room for the whole tensors and each slice's rows (contiguous, starting on
// 16-byte boundaries) are uploaded with that slice, so the first forward
// pass waits only for its own inputs; h0 of batch slices is uploaded whole
// before the first slice, and their final states are gathered whole and
// downloaded after the last slice: fewer, larger copies, each copy having a
// fixed cost on the copy engines.
struct Layout {
  size_t fwd, fwd_bytes, A, D, B, C, h0, fin, carry[2], x[2], dt[2], y[2], total;
};

Layout layout(const ssd_dims &d, ssd_dtype t, const std::vector<Slice> &sl, bool has_D,
              bool has_h0, bool want_fin) {
  Layout l{};
  const size_t e = t == SSD_BF16 ? 2 : 4;
  int64_t nb = 0, nt = 0;
  for (const Slice &s : sl) {
    nb = std::max(nb, s.nb);
    nt = std::max(nt, s.nt);
  }
  const bool seq = d.batch == 1 && sl.size() > 1;
  ssd_dims m = d;
  m.batch = nb;
  m.seqlen = nt;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += r256(bytes);
    return at;
  };
  l.fwd_bytes = ssd_forward_workspace_size(&m, t);
  l.fwd = take(l.fwd_bytes);
  l.A = take(sizeof(float) * d.nheads);
  l.D = take(has_D ? sizeof(float) * d.nheads : 0);
  const size_t state = sizeof(float) * d.nheads * d.headdim * d.dstate;  // one batch row
  const size_t tok = (size_t)d.batch * d.seqlen;
  l.B = take(e * tok * d.ngroups * d.dstate);
  l.C = take(e * tok * d.ngroups * d.dstate);
  l.h0 = take(!seq && has_h0 ? state * d.batch : 0);
  l.fin = take(!seq && want_fin ? state * d.batch : 0);
  for (int p = 0; p < 2; ++p) {
    l.carry[p] = take(seq ? state : 0);
    l.x[p] = take(e * nb * nt * d.nheads * d.headdim);
    l.dt[p] = take(e * nb * nt * d.nheads);
    l.y[p] = take(e * nb * nt * d.nheads * d.headdim);
  }
  l.total = off;
  return l;
}

}  // namespace

extern "C" {

size_t ssd_forward_host_overlapped_workspace_size(const ssd_dims *dims, ssd_dtype dtype,
                                                  int has_D, int has_h0,
                                                  int want_final_state, int n_slices) {
  if (!valid_dims(dims) || (dtype != SSD_F32 && dtype != SSD_BF16) || n_slices < 1) return 0;
  const std::vector<Slice> sl = plan_slices(*dims, n_slices);
  return layout(*dims, dtype, sl, has_D != 0, has_h0 != 0, want_final_state != 0).total;
}

ssd_status ssd_forward_host_overlapped(const ssd_dims *dims, ssd_dtype dtype, const void *x,
                                       const void *dt, const float *A, const void *B,
                                       const void *C, const float *D, const float *h0,
                                       void *y, float *final_state, void *workspace,
                                       size_t ws_bytes, int n_slices, const ssd_plan *plan,
                                       void *stream, void *h2d_stream, void *d2h_stream) {
  // malformed or unsupported dims: the codes ssd_forward gives, nothing enqueued
  if (!valid_dims(dims))
    return ssd_forward(dims, dtype, x, dt, A, B, C, D, h0, y, final_state, nullptr, 0, stream);
  if ((dtype != SSD_F32 && dtype != SSD_BF16) || !x || !dt || !A || !B || !C || !y ||
      !workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || n_slices < 1)
    return SSD_ERR_INVALID_ARG;
  const ssd_dims d = *dims;
  const std::vector<Slice> sl = plan_slices(d, n_slices);
  const bool seq = d.batch == 1 && sl.size() > 1;
  const Layout l = layout(d, dtype, sl, D != nullptr, h0 != nullptr, final_state != nullptr);
  if (ws_bytes < l.total) return SSD_ERR_INVALID_ARG;
  // the plan must suit every slice's dims before anything is enqueued
  for (const Slice &s : sl) {
    ssd_dims sd = d;
    sd.batch = s.nb;
    sd.seqlen = s.nt;
    const ssd_status ps = ssd::plan_status(&sd, dtype, plan);
    if (ps != SSD_OK) return ps;
  }
  char *ws = static_cast<char *>(workspace);
  const size_t e = dtype == SSD_BF16 ? 2 : 4;
  cudaStream_t st = (cudaStream_t)stream;
  cudaStream_t hs = h2d_stream ? (cudaStream_t)h2d_stream : st;
  cudaStream_t ds = d2h_stream ? (cudaStream_t)d2h_stream : st;
  const size_t state = sizeof(float) * d.nheads * d.headdim * d.dstate;
  const int n = (int)sl.size();

  // events: begin, the end of the uploads, the end of the downloads, and per
  // slice: inputs in, forward done, outputs out
  std::vector<cudaEvent_t> ev(3 + 3 * (size_t)n, nullptr);
  cudaError_t err = cudaSuccess;
  for (auto &v : ev)
    if (err == cudaSuccess) err = cudaEventCreateWithFlags(&v, cudaEventDisableTiming);
  auto done_with_events = [&](cudaError_t r) {
    for (auto &v : ev)
      if (v) cudaEventDestroy(v);  // released once recorded work completes
    return r == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
  };
  if (err != cudaSuccess) return done_with_events(err);
  cudaEvent_t ev_begin = ev[0], ev_up_end = ev[1], ev_down_end = ev[2];
  auto ev_in = [&](int i) { return ev[3 + 3 * i]; };
  auto ev_done = [&](int i) { return ev[4 + 3 * i]; };
  auto ev_out = [&](int i) { return ev[5 + 3 * i]; };
  auto ok = [&](cudaError_t r) {
    if (err == cudaSuccess) err = r;
    return err == cudaSuccess;
  };
  auto up = [&](size_t off, const void *src, size_t bytes) {
    if (src && bytes) ok(cudaMemcpyAsync(ws + off, src, bytes, cudaMemcpyHostToDevice, hs));
  };
  auto down = [&](void *dst, size_t off, size_t bytes) {
    if (dst && bytes) ok(cudaMemcpyAsync(dst, ws + off, bytes, cudaMemcpyDeviceToHost, ds));
  };

  ok(cudaEventRecord(ev_begin, st));
  if (hs != st) ok(cudaStreamWaitEvent(hs, ev_begin, 0));
  if (ds != st) ok(cudaStreamWaitEvent(ds, ev_begin, 0));
  up(l.A, A, sizeof(float) * d.nheads);
  up(l.D, D, sizeof(float) * d.nheads);
  if (seq)
    up(l.carry[0], h0, state);
  else
    up(l.h0, h0, state * d.batch);
  ssd_status status = SSD_OK;
  for (int i = 0; i < n && err == cudaSuccess && status == SSD_OK; ++i) {
    const Slice &s = sl[i];
    const int p = i & 1;
    // inputs of slice i (its buffer is free once forward i - 2 is done)
    if (i >= 2) ok(cudaStreamWaitEvent(hs, ev_done(i - 2), 0));
    const int64_t tok0 = s.b0 * d.seqlen + s.t0, ntok = s.nb * s.nt;
    up(l.x[p], static_cast<const char *>(x) + e * tok0 * d.nheads * d.headdim,
       e * ntok * d.nheads * d.headdim);
    up(l.dt[p], static_cast<const char *>(dt) + e * tok0 * d.nheads, e * ntok * d.nheads);
    const size_t bc_off = e * tok0 * d.ngroups * d.dstate, bc_len = e * ntok * d.ngroups * d.dstate;
    up(l.B + bc_off, static_cast<const char *>(B) + bc_off, bc_len);
    up(l.C + bc_off, static_cast<const char *>(C) + bc_off, bc_len);
    ok(cudaEventRecord(ev_in(i), hs));
    // forward of slice i (its y buffer is free once the download of slice
    // i - 2 is done)
    ok(cudaStreamWaitEvent(st, ev_in(i), 0));
    if (i >= 2) ok(cudaStreamWaitEvent(st, ev_out(i - 2), 0));
    if (err != cudaSuccess) break;
    ssd_dims sd = d;
    sd.batch = s.nb;
    sd.seqlen = s.nt;
    const float *h_in =
        seq ? ((i == 0 && !h0) ? nullptr : reinterpret_cast<const float *>(ws + l.carry[p]))
            : (h0 ? reinterpret_cast<const float *>(ws + l.h0 + s.b0 * state) : nullptr);
    float *h_out = seq ? reinterpret_cast<float *>(ws + l.carry[p ^ 1])
                       : (final_state ? reinterpret_cast<float *>(ws + l.fin + s.b0 * state)
                                      : nullptr);
    // the forward's workspace sits at offset 0: its error word is this
    // workspace's
    status = ssd_forward_ex(&sd, dtype, ws + l.x[p], ws + l.dt[p],
                            reinterpret_cast<const float *>(ws + l.A),
                            ws + l.B + e * tok0 * d.ngroups * d.dstate,
                            ws + l.C + e * tok0 * d.ngroups * d.dstate,
                            D ? reinterpret_cast<const float *>(ws + l.D) : nullptr, h_in,
                            ws + l.y[p], h_out, ws + l.fwd, l.fwd_bytes, plan, stream);
    ok(cudaEventRecord(ev_done(i), st));
    // outputs of slice i
    ok(cudaStreamWaitEvent(ds, ev_done(i), 0));
    down(static_cast<char *>(y) + e * tok0 * d.nheads * d.headdim, l.y[p],
         e * ntok * d.nheads * d.headdim);
    if (i == n - 1) {
      if (seq)
        down(final_state, l.carry[p ^ 1], state);
      else
        down(final_state, l.fin, state * d.batch);
    }
    ok(cudaEventRecord(ev_out(i), ds));
  }
  // The caller's stream is ordered after everything enqueued on the two copy
  // streams -- also when a step above failed, so that the caller never frees
  // or reuses the host buffers or the workspace while a copy already queued
  // is still running.  Each join is attempted whatever happened before.
  cudaError_t jerr = cudaSuccess;
  auto join = [&](cudaStream_t from, cudaEvent_t evt) {
    if (from == st) return;
    cudaError_t r = cudaEventRecord(evt, from);
    if (r == cudaSuccess) r = cudaStreamWaitEvent(st, evt, 0);
    if (jerr == cudaSuccess) jerr = r;
  };
  join(hs, ev_up_end);
  join(ds, ev_down_end);
  if (err == cudaSuccess) err = jerr;
  const ssd_status r = done_with_events(err);
  return status != SSD_OK ? status : r;
}

}  // extern "C"
