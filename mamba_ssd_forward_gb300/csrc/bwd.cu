// Backward pass of the chunked SSD (fp32 I/O): the gradients of a loss L
// through the forward recurrence of "Accelerating Mamba-2 with
// High-Performance Forward Pass Kernels in NVIDIA CUDA Tile", section
// "Mamba-2 architecture" (h_t = a_t h_{t-1} + dt_t x_t B_t^T, y_t = h_t c_t +
// D x_t), given gy = dL/dy and gfinal = dL/dfinal_state.  The pages name the
// backward pass but do not derive it; the chunked formulas below follow from
// the adjoint recurrence g_t = gy_t c_t^T + a_{t+1} g_{t+1}.  Per (batch,
// head), with G the inclusive in-chunk cumsum of l_t = A dt_t (log2 units
// here), h_k the state entering chunk k and R_k = dL/dh_{k+1} arriving from
// the chunks after k (R of the last chunk = gfinal):
//
//   R_{k-1} = exp2(G_last) R_k + sum_{s in k} exp2(G_s) gy_s c_s^T   (dh0 = R_{-1})
//   dx_t  = dt_t [sum_{s>=t} exp2(G_s - G_t) (B_t . C_s) gy_s + exp2(G_last - G_t) R_k B_t] + D gy_t
//   q_t   = sum_{s>=t} exp2(G_s - G_t) (gy_s . x_t) C_s + exp2(G_last - G_t) R_k^T x_t
//   dB_t += dt_t q_t,   dC_t += exp2(G_t) h_k^T gy_t + sum_{j<=t} exp2(G_t - G_j) (gy_t . x_j) dt_j B_j
//   ysm_t = exp2(G_t) h_k c_t + sum_{j<=t} exp2(G_t - G_j) (c_t . B_j) dt_j x_j     (y - D x)
//   dL/dG_i = gy_i . ysm_i - x_i . (dx_i - D gy_i)  (+ <R_k, h_{k+1}> at the chunk's last token)
//   eta_t = sum_{i>=t in k} dL/dG_i  (= dL/dl_t, natural-log units)
//   ddt_t = A eta_t + q_t . B_t,   dA = sum_t dt_t eta_t,   dD = sum_t gy_t . x_t
//
// (dB and dC sum over the heads of a group.)  The forward's cumsum kernel
// gives G; then:
//   bwd_jump_kernel   the forward's chunk jump terms sum_j exp2(G_last - G_j)
//                     dt_j x_j B_j^T in fp32 (the forward's own kernels take
//                     TF32 products, whose rounding the sums through
//                     <R_k, h_{k+1}> into dA would carry at about 3e-3);
//   state_passing     forwards over the chunks for h_k and the final state;
//   bwd_jump_kernel   the adjoint's chunk jump terms sum_s exp2(G_s) gy_s c_s^T;
//   state_passing     backwards over the chunks for R_k and dh0;
//   bwd_main_kernel   per (batch, head, chunk, 32-token tile): dx, q, the
//                     head's share of dC, and per token q . B, dL/dG, gy . x;
//   bwd_finish_kernel per (batch, head, chunk): the reverse cumsum for eta,
//                     ddt, and the chunk's shares of dA and dD;
//   bwd_reduce_kernel the sums over the heads of a group (dB, dC) and over
//                     batches and chunks (dA, dD), in a fixed order.
// All in fp32 on the CUDA cores (the tensor-core version is the next step):
// about 30 million multiply-adds per chunk and head at T = 256, P = 64,
// S = 128.
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kTT = 32;  // tokens per tile of bwd_main_kernel
constexpr int kP = 64;

// ---------------------------------------------------------------- jump terms

// out[b, h, k][p][s] = sum_{t in chunk k} w_t v_t[p] m_t[s], v per head
// ([b, L, nh, P]) and m per group ([b, L, ng, S]): the adjoint's jump terms
// (v = gy, m = C, w_t = exp2(G_t); dt null) or the forward's (v = x, m = B,
// w_t = exp2(G_last - G_t) dt_t).  One CTA per (chunk, batch * head),
// thread = kS / 4 outputs (e = tid + 256 i: p = e / S, s = e % S; a warp's
// lanes share p and read consecutive s).
template <int kS>
__global__ void __launch_bounds__(kThreads)
bwd_jump_kernel(const float *__restrict__ v, const float *__restrict__ m,
                const float *__restrict__ dt, const float *__restrict__ G,
                float *__restrict__ out, int *err, int L, int nh, int hpg, int T, int nc,
                int nb) {
  constexpr int kPer = kP * kS / kThreads;
  const int ng = nh / hpg;
  __shared__ float gys[kTT][kP];
  __shared__ float cs[kTT][kS];
  const int k = blockIdx.x, bh = blockIdx.y;
  const int b = bh / nh, h = bh - b * nh, g = h / hpg;
  const int tok0 = k * T, valid = min(T, L - tok0);
  const int tid = threadIdx.x;
  if (!SSD_IN_BOUNDS(b < nb && k < nc, err, 200)) return;  // uniform over the CTA
  float acc[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
  const float *Gc = G + ((int64_t)bh * nc + k) * T;
  const float Glast = Gc[valid - 1];
  for (int t0 = 0; t0 < valid; t0 += kTT) {
    __syncthreads();
    for (int e = tid; e < kTT * kP; e += kThreads) {
      const int tt = e / kP, p = e % kP, t = t0 + tt;
      float w = 0.f;
      if (t < valid) {
        const int64_t tok = (int64_t)b * L + tok0 + t;
        w = dt ? exp2f(Glast - Gc[t]) * dt[tok * nh + h] : exp2f(Gc[t]);
        w *= v[(tok * nh + h) * kP + p];
      }
      gys[tt][p] = w;
    }
    for (int e = tid; e < kTT * kS; e += kThreads) {
      const int tt = e / kS, s = e % kS, t = t0 + tt;
      cs[tt][s] = t < valid ? m[(((int64_t)b * L + tok0 + t) * ng + g) * kS + s] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int tt = 0; tt < kTT; ++tt) {
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int e = tid + kThreads * i;
        acc[i] = fmaf(gys[tt][e / kS], cs[tt][e % kS], acc[i]);
      }
    }
  }
  float *dst = out + ((int64_t)bh * nc + k) * kP * kS;
#pragma unroll
  for (int i = 0; i < kPer; ++i) dst[tid + kThreads * i] = acc[i];
}

// -------------------------------------------------------------- main kernel

// One CTA per (32-token tile of a chunk, chunk, batch * head); thread = (token
// tt = tid / 8 of the tile, lane l8 = tid % 8), the lane holding columns
// l8 + 8 m of its token's outputs and the 8 lanes of a token splitting every
// dot product.  Shared memory (row strides padded by one float): the tile's
// B, C, x, gy; one other tile at a time (C and gy for the s >= t sums, B and
// x for the j <= t sums); the chunk's G and dt; R_k, then h_k, as [P][S].
template <int kS>
__global__ void __launch_bounds__(kThreads)
bwd_main_kernel(const float *__restrict__ x, const float *__restrict__ dt,
                const float *__restrict__ Bm, const float *__restrict__ Cm,
                const float *__restrict__ D, const float *__restrict__ gy,
                const float *__restrict__ G, const float *__restrict__ states,
                const float *__restrict__ R, float *__restrict__ dx,
                float *__restrict__ dBh, float *__restrict__ dCh, float *__restrict__ qB,
                float *__restrict__ dG, float *__restrict__ gyx, int *err, int L, int nh,
                int hpg, int T, int nc, int nb) {
  constexpr int SP = kS + 1, PP = kP + 1;
  constexpr int kMS = kS / 8, kMP = kP / 8;
  extern __shared__ float sm[];
  float *Bt = sm;                 // [32][SP]
  float *Ct = Bt + kTT * SP;      // [32][SP]
  float *xt = Ct + kTT * SP;      // [32][PP]
  float *gt = xt + kTT * PP;      // [32][PP]
  float *U1 = gt + kTT * PP;      // [32][SP]  other tile: C (upper) or B (lower)
  float *U2 = U1 + kTT * SP;      // [32][PP]  other tile: gy (upper) or x (lower)
  float *Gs = U2 + kTT * PP;      // [256]
  float *ds = Gs + 256;           // [256]
  float *M = ds + 256;            // [64][SP]  R_k, then h_k

  const int ntile = T / kTT;
  const int k = blockIdx.x / ntile, tau = blockIdx.x - k * ntile;
  const int bh = blockIdx.y, b = bh / nh, h = bh - b * nh, g = h / hpg, ng = nh / hpg;
  const int tok0 = k * T, valid = min(T, L - tok0);
  const int tid = threadIdx.x, tt = tid >> 3, l8 = tid & 7;
  if (!SSD_IN_BOUNDS(b < nb && k < nc, err, 201)) return;  // uniform over the CTA
  if (tau * kTT >= valid) return;                           // tile past the sequence
  const int t = tau * kTT + tt;                             // chunk-relative token
  const bool live = t < valid;

  auto row_x = [&](int tok) { return (((int64_t)b * L + tok0 + tok) * nh + h) * kP; };
  auto row_g = [&](int tok) { return (((int64_t)b * L + tok0 + tok) * ng + g) * kS; };
  // load a 32-token tile of a [b, L, (heads or groups), width] tensor into a
  // padded shared array (zeros past the sequence)
  auto load_tile = [&](float *dst, int stride, const float *src, int width, bool per_head,
                       int u) {
    for (int e = tid; e < kTT * width; e += kThreads) {
      const int r = e / width, c = e - r * width, tok = u * kTT + r;
      float v = 0.f;
      if (tok < valid) v = src[(per_head ? row_x(tok) : row_g(tok)) + c];
      dst[r * stride + c] = v;
    }
  };
  const float *Gc = G + ((int64_t)bh * nc + k) * T;
  for (int i = tid; i < T; i += kThreads) {
    Gs[i] = Gc[i];
    ds[i] = i < valid ? dt[((int64_t)b * L + tok0 + i) * nh + h] : 0.f;
  }
  load_tile(Bt, SP, Bm, kS, false, tau);
  load_tile(Ct, SP, Cm, kS, false, tau);
  load_tile(xt, PP, x, kP, true, tau);
  load_tile(gt, PP, gy, kP, true, tau);
  __syncthreads();
  const float Gt = Gs[min(t, T - 1)], dtt = ds[min(t, T - 1)];
  const float GL = Gs[valid - 1];

  float dxs[kMP], ysm[kMP], q[kMS], dc[kMS];
#pragma unroll
  for (int m = 0; m < kMP; ++m) dxs[m] = ysm[m] = 0.f;
#pragma unroll
  for (int m = 0; m < kMS; ++m) q[m] = dc[m] = 0.f;
  // the dot product of this token's row a and row j of b over a width, split
  // over the 8 lanes of the token
  auto dot8 = [&](const float *a, const float *bb, int width) {
    float s = 0.f;
    for (int c = l8; c < width; c += 8) s = fmaf(a[c], bb[c], s);
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    s += __shfl_xor_sync(0xffffffffu, s, 4);
    return s;
  };

  // s >= t: dx += dt_t exp2(G_s - G_t) (B_t . C_s) gy_s,  q += exp2(G_s - G_t) (gy_s . x_t) C_s
  for (int u = tau; u < ntile && u * kTT < valid; ++u) {
    __syncthreads();
    load_tile(U1, SP, Cm, kS, false, u);
    load_tile(U2, PP, gy, kP, true, u);
    __syncthreads();
    for (int j = 0; j < kTT; ++j) {
      const int s = u * kTT + j;
      const float S1 = dot8(Bt + tt * SP, U1 + j * SP, kS);
      const float X1 = dot8(xt + tt * PP, U2 + j * PP, kP);
      const float w = (s >= t && s < valid && live) ? exp2f(Gs[s] - Gt) : 0.f;
      const float a1 = dtt * w * S1, b1 = w * X1;
#pragma unroll
      for (int m = 0; m < kMP; ++m) dxs[m] = fmaf(a1, U2[j * PP + l8 + 8 * m], dxs[m]);
#pragma unroll
      for (int m = 0; m < kMS; ++m) q[m] = fmaf(b1, U1[j * SP + l8 + 8 * m], q[m]);
    }
  }
  // j <= t: ysm += exp2(G_t - G_j) dt_j (c_t . B_j) x_j,  dC += exp2(G_t - G_j) dt_j (gy_t . x_j) B_j
  for (int u = 0; u <= tau; ++u) {
    __syncthreads();
    load_tile(U1, SP, Bm, kS, false, u);
    load_tile(U2, PP, x, kP, true, u);
    __syncthreads();
    for (int j = 0; j < kTT; ++j) {
      const int jj = u * kTT + j;
      const float S2 = dot8(Ct + tt * SP, U1 + j * SP, kS);
      const float X2 = dot8(gt + tt * PP, U2 + j * PP, kP);
      const float w = (jj <= t && jj < valid && live) ? exp2f(Gt - Gs[jj]) * ds[jj] : 0.f;
      const float a2 = w * S2, b2 = w * X2;
#pragma unroll
      for (int m = 0; m < kMP; ++m) ysm[m] = fmaf(a2, U2[j * PP + l8 + 8 * m], ysm[m]);
#pragma unroll
      for (int m = 0; m < kMS; ++m) dc[m] = fmaf(b2, U1[j * SP + l8 + 8 * m], dc[m]);
    }
  }
  // state terms: R_k (dx: R B_t; q: R^T x_t), then h_k (ysm: h c_t; dC: h^T gy_t)
  const int64_t st_row = ((int64_t)bh * nc + k) * kP * kS;
  for (int pass = 0; pass < 2; ++pass) {
    __syncthreads();
    const float *src = pass == 0 ? R + st_row : states + st_row;
    for (int e = tid; e < kP * kS; e += kThreads) M[(e / kS) * SP + e % kS] = src[e];
    __syncthreads();
    const float fa = pass == 0 ? (live ? dtt * exp2f(GL - Gt) : 0.f) : (live ? exp2f(Gt) : 0.f);
    const float fb = pass == 0 ? (live ? exp2f(GL - Gt) : 0.f) : fa;
    const float *va = pass == 0 ? Bt + tt * SP : Ct + tt * SP;  // [S]
    const float *vb = pass == 0 ? xt + tt * PP : gt + tt * PP;  // [P]
#pragma unroll
    for (int m = 0; m < kMP; ++m) {  // rows p = l8 + 8 m: M[p] . va
      const float *row = M + (l8 + 8 * m) * SP;
      float s = 0.f;
      for (int c = 0; c < kS; ++c) s = fmaf(row[c], va[c], s);
      if (pass == 0)
        dxs[m] = fmaf(fa, s, dxs[m]);
      else
        ysm[m] = fmaf(fa, s, ysm[m]);
    }
#pragma unroll
    for (int m = 0; m < kMS; ++m) {  // columns s = l8 + 8 m: M[:, s] . vb
      float s = 0.f;
      for (int p = 0; p < kP; ++p) s = fmaf(M[p * SP + l8 + 8 * m], vb[p], s);
      if (pass == 0)
        q[m] = fmaf(fb, s, q[m]);
      else
        dc[m] = fmaf(fb, s, dc[m]);
    }
  }
  // outputs of this token
  const float Dh = D ? D[h] : 0.f;
  float gdot = 0.f, xdot = 0.f, qb = 0.f, gx = 0.f;
#pragma unroll
  for (int m = 0; m < kMP; ++m) {
    const int p = l8 + 8 * m;
    gdot = fmaf(gt[tt * PP + p], ysm[m], gdot);
    xdot = fmaf(xt[tt * PP + p], dxs[m], xdot);
    gx = fmaf(gt[tt * PP + p], xt[tt * PP + p], gx);
  }
#pragma unroll
  for (int m = 0; m < kMS; ++m) qb = fmaf(q[m], Bt[tt * SP + l8 + 8 * m], qb);
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    gdot += __shfl_xor_sync(0xffffffffu, gdot, o);
    xdot += __shfl_xor_sync(0xffffffffu, xdot, o);
    qb += __shfl_xor_sync(0xffffffffu, qb, o);
    gx += __shfl_xor_sync(0xffffffffu, gx, o);
  }
  if (!live) return;  // no barrier follows
  const int64_t rx = row_x(t);
#pragma unroll
  for (int m = 0; m < kMP; ++m) {
    const int p = l8 + 8 * m;
    dx[rx + p] = dxs[m] + Dh * gt[tt * PP + p];
  }
  const int64_t rs = (((int64_t)b * L + tok0 + t) * nh + h) * kS;
#pragma unroll
  for (int m = 0; m < kMS; ++m) {
    dBh[rs + l8 + 8 * m] = dtt * q[m];
    dCh[rs + l8 + 8 * m] = dc[m];
  }
  if (l8 == 0) {
    const int64_t o = ((int64_t)bh * nc + k) * T + t;
    qB[o] = qb;
    dG[o] = gdot - xdot;
    gyx[o] = gx;
  }
}

// ------------------------------------------------------------ finish (eta)

// One CTA per (chunk, batch * head), thread = token: <R_k, h_{k+1}> joins dL/dG
// at the chunk's last real token, eta is the reverse cumsum over the chunk,
// ddt = A eta + q . B; the chunk's shares of dA and dD go to part[] (reduced
// in a fixed order later).  eta is a sum of gradients with respect to the
// natural-log cumsum, whatever units G is kept in.
__global__ void __launch_bounds__(kThreads)
bwd_finish_kernel(const float *__restrict__ dt, const float *__restrict__ A,
                  const float *__restrict__ R, const float *__restrict__ states,
                  const float *__restrict__ final_state, const float *__restrict__ qB,
                  const float *__restrict__ dG, const float *__restrict__ gyx,
                  float *__restrict__ ddt, float2 *__restrict__ part, int *err, int L, int nh,
                  int P, int S, int T, int nc, int nb) {
  __shared__ float red[kThreads / 32];
  __shared__ float tot[kThreads / 32];
  const int k = blockIdx.x, bh = blockIdx.y, b = bh / nh, h = bh - b * nh;
  const int tok0 = k * T, valid = min(T, L - tok0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (!SSD_IN_BOUNDS(b < nb && k < nc, err, 202)) return;  // uniform over the CTA
  // <R_k, h_{k+1}> over P x S
  const float *Rk = R + ((int64_t)bh * nc + k) * P * S;
  const float *hn = k + 1 < nc ? states + ((int64_t)bh * nc + k + 1) * P * S
                               : final_state + (int64_t)bh * P * S;
  float s = 0.f;
  for (int e = tid; e < P * S; e += kThreads) s = fmaf(Rk[e], hn[e], s);
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) red[warp] = s;
  __syncthreads();
  float rh = 0.f;
  for (int w = 0; w < kThreads / 32; ++w) rh += red[w];
  // reverse inclusive cumsum of dL/dG over the chunk's tokens (thread = token)
  const int64_t o = ((int64_t)bh * nc + k) * T + tid;
  float v = 0.f;
  if (tid < valid) v = dG[o] + (tid == valid - 1 ? rh : 0.f);
  // suffix sums: scan the reversed order within the warp, then across warps
  float incl = v;
  for (int off = 1; off < 32; off <<= 1) {
    const float nb2 = __shfl_down_sync(0xffffffffu, incl, off);
    if (lane + off < 32) incl += nb2;
  }
  if (lane == 0) tot[warp] = incl;  // the warp's total
  __syncthreads();
  float after = 0.f;  // totals of the warps after this one
  for (int w = warp + 1; w < kThreads / 32; ++w) after += tot[w];
  const float eta = incl + after;
  float dA_part = 0.f, dD_part = 0.f;
  if (tid < valid) {
    const float dtt = dt[((int64_t)b * L + tok0 + tid) * nh + h];
    ddt[((int64_t)b * L + tok0 + tid) * nh + h] = A[h] * eta + qB[o];
    dA_part = dtt * eta;
    dD_part = gyx[o];
  }
  for (int off = 16; off > 0; off >>= 1) {
    dA_part += __shfl_xor_sync(0xffffffffu, dA_part, off);
    dD_part += __shfl_xor_sync(0xffffffffu, dD_part, off);
  }
  __syncthreads();
  if (lane == 0) {
    red[warp] = dA_part;
    tot[warp] = dD_part;
  }
  __syncthreads();
  if (tid == 0) {
    float a = 0.f, d = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) {
      a += red[w];
      d += tot[w];
    }
    part[(int64_t)bh * nc + k] = make_float2(a, d);
  }
}

// ------------------------------------------------------------------ reduce

// dB[b, t, g, s] = sum over the group's heads of dBh[b, t, h, s] (same for
// dC), one thread per output element (none when each group has one head:
// bwd_main then writes dB and dC itself); then (threads past those) dA and
// dD per head over batches and chunks, in a fixed order.
__global__ void __launch_bounds__(kThreads)
bwd_reduce_kernel(const float *__restrict__ dBh, const float *__restrict__ dCh,
                  const float2 *__restrict__ part, float *__restrict__ dB,
                  float *__restrict__ dC, float *__restrict__ dA, float *__restrict__ dD,
                  int64_t n_bc, int nh, int hpg, int S, int nc, int nb) {
  const int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int ng = nh / hpg;
  if (e < n_bc) {
    const int s = (int)(e % S);
    const int64_t r = e / S;  // (b, t, g)
    const int g = (int)(r % ng);
    const int64_t bt = r / ng;
    float sb = 0.f, sc = 0.f;
    for (int i = 0; i < hpg; ++i) {
      const int64_t src = (bt * nh + g * hpg + i) * S + s;
      sb += dBh[src];
      sc += dCh[src];
    }
    dB[e] = sb;
    dC[e] = sc;
  } else if (e - n_bc < nh) {
    const int h = (int)(e - n_bc);
    float a = 0.f, d = 0.f;
    for (int b = 0; b < nb; ++b)
      for (int k = 0; k < nc; ++k) {
        const float2 v = part[((int64_t)b * nh + h) * nc + k];
        a += v.x;
        d += v.y;
      }
    dA[h] = a;
    if (dD) dD[h] = d;
  }
}

}  // namespace

bool bwd_supported(const Dims &d) {
  return d.P == kP && (d.S == 64 || d.S == 128 || d.S == 256) && d.T % kTT == 0 && d.T <= 256;
}

size_t bwd_main_smem(const Dims &d) {
  const int SP = (int)d.S + 1, PP = kP + 1;
  return sizeof(float) * (size_t)(3 * kTT * SP + 3 * kTT * PP + 512 + 64 * SP);
}

cudaError_t launch_bwd_jump(const Dims &d, const float *v, const float *m, const float *dt,
                            const float *G, float *out, int *err, cudaStream_t st) {
  dim3 grid((unsigned)d.nc, (unsigned)(d.b * d.nh));
  const int L = (int)d.L, nh = (int)d.nh, hpg = (int)d.hpg, T = (int)d.T, nc = (int)d.nc,
            nb = (int)d.b;
  switch (d.S) {
    case 64: bwd_jump_kernel<64><<<grid, kThreads, 0, st>>>(v, m, dt, G, out, err, L, nh, hpg, T, nc, nb); break;
    case 128: bwd_jump_kernel<128><<<grid, kThreads, 0, st>>>(v, m, dt, G, out, err, L, nh, hpg, T, nc, nb); break;
    default: bwd_jump_kernel<256><<<grid, kThreads, 0, st>>>(v, m, dt, G, out, err, L, nh, hpg, T, nc, nb); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_main(const Dims &d, const float *x, const float *dt, const float *B,
                            const float *C, const float *D, const float *gy, const float *G,
                            const float *states, const float *R, float *dx, float *dBh,
                            float *dCh, float *qB, float *dG, float *gyx, int *err,
                            cudaStream_t st) {
  dim3 grid((unsigned)(d.nc * (d.T / kTT)), (unsigned)(d.b * d.nh));
  const size_t smem = bwd_main_smem(d);
  const int L = (int)d.L, nh = (int)d.nh, hpg = (int)d.hpg, T = (int)d.T, nc = (int)d.nc,
            nb = (int)d.b;
  cudaError_t e = cudaSuccess;
  switch (d.S) {
    case 64:
      e = cudaFuncSetAttribute(bwd_main_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
      if (e == cudaSuccess)
        bwd_main_kernel<64><<<grid, kThreads, smem, st>>>(x, dt, B, C, D, gy, G, states, R, dx,
                                                          dBh, dCh, qB, dG, gyx, err, L, nh,
                                                          hpg, T, nc, nb);
      break;
    case 128:
      e = cudaFuncSetAttribute(bwd_main_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
      if (e == cudaSuccess)
        bwd_main_kernel<128><<<grid, kThreads, smem, st>>>(x, dt, B, C, D, gy, G, states, R, dx,
                                                           dBh, dCh, qB, dG, gyx, err, L, nh,
                                                           hpg, T, nc, nb);
      break;
    default:
      e = cudaFuncSetAttribute(bwd_main_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
      if (e == cudaSuccess)
        bwd_main_kernel<256><<<grid, kThreads, smem, st>>>(x, dt, B, C, D, gy, G, states, R, dx,
                                                           dBh, dCh, qB, dG, gyx, err, L, nh,
                                                           hpg, T, nc, nb);
      break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_bwd_finish(const Dims &d, const float *dt, const float *A, const float *R,
                              const float *states, const float *final_state, const float *qB,
                              const float *dG, const float *gyx, float *ddt, float2 *part,
                              int *err, cudaStream_t st) {
  dim3 grid((unsigned)d.nc, (unsigned)(d.b * d.nh));
  bwd_finish_kernel<<<grid, kThreads, 0, st>>>(dt, A, R, states, final_state, qB, dG, gyx, ddt,
                                               part, err, (int)d.L, (int)d.nh, (int)d.P,
                                               (int)d.S, (int)d.T, (int)d.nc, (int)d.b);
  return cudaGetLastError();
}

cudaError_t launch_bwd_reduce(const Dims &d, const float *dBh, const float *dCh,
                              const float2 *part, float *dB, float *dC, float *dA, float *dD,
                              cudaStream_t st) {
  const int64_t n_bc = d.hpg > 1 ? d.b * d.L * d.ng * d.S : 0;
  const int64_t n = n_bc + d.nh;
  bwd_reduce_kernel<<<(unsigned)((n + kThreads - 1) / kThreads), kThreads, 0, st>>>(
      dBh, dCh, part, dB, dC, dA, dD, n_bc, (int)d.nh, (int)d.hpg, (int)d.S, (int)d.nc,
      (int)d.b);
  return cudaGetLastError();
}

}  // namespace ssd
