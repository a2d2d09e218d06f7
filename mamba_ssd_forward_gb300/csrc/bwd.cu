// Backward pass of the chunked SSD (fp32 arithmetic): the gradients of a loss L
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
//   bwd_scale_kernel  x~ = dt_t exp2(G_last - G_t) x_t, gy~ = exp2(G_t) gy_t;
//   bwd_state_gemm    (bwd_gemm.cu, split-TF32 tensor-core GEMMs) the
//                     forward's chunk jump terms sum_j x~_j B_j^T (the
//                     forward's own kernels take plain TF32 products, whose
//                     rounding the sums through <R_k, h_{k+1}> into dA would
//                     carry at about 3e-3);
//   state_passing     forwards over the chunks for h_k and the final state;
//   bwd_state_gemm    the adjoint's chunk jump terms sum_s gy~_s c_s^T;
//   state_passing     backwards over the chunks for R_k and dh0;
//   bwd_state_gemm    c_i . B_j of every chunk and group (Kcb);
//   bwd_state_gemm    the state terms R_k B_t and h_k c_t per token and head;
//   bwd_main_kernel   per (row tile, chunk, batch * group), walking the
//                     group's heads: dx of each head and per token q . B,
//                     dL/dG, gy . x, and the group's dB and dC, the S-side
//                     weights summed over the heads before one update;
//   bwd_finish_kernel per (batch, head, chunk): the reverse cumsum for eta,
//                     ddt, and the chunk's shares of dA and dD;
//   bwd_reduce_kernel dB, dC summed over head slices (when a group's heads
//                     are split over CTAs), and the sums over batches and
//                     chunks (dA, dD), in a fixed order;
//   bwd_state_gemm    dB += x~ R_k, dC += gy~ h_k (summed over the group's heads);
//   bwd_convert_kernel with bf16 I/O, the inputs to fp32 copies before and
//                     the gradients back to bf16 after.
// The kernels of this file run in fp32 on the CUDA cores (plain TF32
// tensor-core products would put dA off by about 1 %), the state terms'
// GEMMs in split TF32 on the tensor cores.

#include <algorithm>
#include <cstdint>
#include <type_traits>

#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kTT = 32;  // tokens per tile of bwd_main_kernel
constexpr int kP = 64;

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool full) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem),
               "r"(full ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ float dot4(const float4 &a, const float4 &b, float s) {
  s = fmaf(a.x, b.x, s);
  s = fmaf(a.y, b.y, s);
  s = fmaf(a.z, b.z, s);
  return fmaf(a.w, b.w, s);
}
__device__ __forceinline__ void axpy4(float a, const float4 &v, float4 &acc) {
  acc.x = fmaf(a, v.x, acc.x);
  acc.y = fmaf(a, v.y, acc.y);
  acc.z = fmaf(a, v.z, acc.z);
  acc.w = fmaf(a, v.w, acc.w);
}
__device__ __forceinline__ float comp(const float4 &v, int e) {
  return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}

// ------------------------------------------------------------ state terms

// The token-row operands of the backward's GEMMs (bwd_gemm.cu) that carry
// a per-token factor: X~ = dt exp2(G_last - G_t) x (the forward's jump
// terms, dB += X~ R) and Gy~ = exp2(G_t) gy (the adjoint's jump terms, dC
// += Gy~ h), in the layout of x, one thread per four elements of [b, L, nh,
// P].  (Applying the factors inside the GEMM's split instead was measured
// slower on the long-context layer: the factor loads land on the GEMM's
// critical path.)
__global__ void __launch_bounds__(kThreads)
bwd_scale_kernel(const float *__restrict__ x, const float *__restrict__ gy,
                 const float *__restrict__ dt, const float *__restrict__ G,
                 float *__restrict__ xs, float *__restrict__ gys, int *err, int L, int nh,
                 int T, int nc, int nb) {
  constexpr int P4 = kP / 4;
  const int64_t n4 = (int64_t)nb * L * nh * P4;
  for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < n4;
       e += (int64_t)gridDim.x * kThreads) {
    const int64_t rowh = e / P4;  // (b * L + t) * nh + h
    const int h = (int)(rowh % nh);
    const int64_t tok = rowh / nh;
    const int b = (int)(tok / L), t = (int)(tok - (int64_t)b * L);
    const int k = t / T, tt = t - k * T, valid = min(T, L - k * T);
    const float *Gc = G + (((int64_t)b * nh + h) * nc + k) * T;
    const float Gt = Gc[tt], GL = Gc[valid - 1];
    const float fx = dt[rowh] * exp2f(GL - Gt), fg = exp2f(Gt);
    if (!SSD_IN_BOUNDS(e < n4, err, 220)) continue;
    const float4 xv = reinterpret_cast<const float4 *>(x)[e];
    const float4 gv = reinterpret_cast<const float4 *>(gy)[e];
    reinterpret_cast<float4 *>(xs)[e] = make_float4(fx * xv.x, fx * xv.y, fx * xv.z, fx * xv.w);
    reinterpret_cast<float4 *>(gys)[e] = make_float4(fg * gv.x, fg * gv.y, fg * gv.z, fg * gv.w);
  }
}

// -------------------------------------------------------------- main kernel


// Sums each of the V values v[] over the kG lanes of a token group (the
// lanes that differ in their low log2(kG) bits; `lane` is the lane of the
// warp, kG divides 32) and leaves every total in every lane: a reduce-scatter (at the step with lane bit o a lane keeps one
// half of its values, adds the partner's copy of that half, and passes on
// the other half), the remaining steps on the single value left, and a
// gather of the V totals from the lanes holding them.  2V - 1 + log2(kG / V)
// shuffles instead of V log2(kG).
template <int V, int kG>
__device__ __forceinline__ void group_sums(float (&v)[V], int lane) {
  static_assert(V >= 1 && V <= kG && (V & (V - 1)) == 0, "V: a power of two up to kG");
  int idx = 0;  // index (into v) of the total this lane ends up holding
#pragma unroll
  for (int n = V, o = 1; n > 1; n >>= 1, o <<= 1) {
    const bool up = lane & o;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float keep = up ? v[i + n / 2] : v[i], send = up ? v[i] : v[i + n / 2];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
    if (up) idx += n / 2;
  }
#pragma unroll
  for (int o = V; o < kG; o <<= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
  // lane (lane & ~(V - 1)) | m holds total idx(m): bit o of m (o = 1, 2, ..)
  // adds V / 2o; gather every total from one such lane of this group
  const float mine = v[0];
  (void)idx;
#pragma unroll
  for (int k = 0; k < V; ++k) {
    int m = 0;
#pragma unroll
    for (int n = V, o = 1; n > 1; n >>= 1, o <<= 1)
      if (k & (n / 2)) m |= o;
    v[k] = __shfl_sync(0xffffffffu, mine, (lane & ~(V - 1)) | m);
  }
}

// Sums each of the kG values v[] over the kG lanes of a token group and
// leaves one total in each lane: the reduce-scatter of group_sums (kG - 1
// shuffles).  Returns the total; *idx = the index (into v) it belongs to.
template <int kG>
__device__ __forceinline__ float group_scatter(float (&v)[kG], int lane, int *idx) {
  int id = 0;
#pragma unroll
  for (int n = kG, o = 1; n > 1; n >>= 1, o <<= 1) {
    const bool up = lane & o;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float keep = up ? v[i + n / 2] : v[i], send = up ? v[i] : v[i + n / 2];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
    if (up) id += n / 2;
  }
  *idx = id;
  return v[0];
}


// Shared-memory plan of bwd_main_kernel (float4 units unless noted):
//   Wsum [RT][WR] floats  the S-side weights of the pass summed over the
//                         group's heads (WR = 256 + 4)
//   U2   [2][NT][P/4]     a head's P-wide column tiles (gy upper, x lower)
//   Kt   [2] x KT4        the c . B block of the tile pair ([NT][RT + 4]
//                         floats in the upper pass, [RT][NT + 4] in the lower)
//   Wt   [RT][NT + 4]     floats: a head's P-side weights of one tile
//   Qp   [RT][CB]         floats: the lanes' shares of q . B (upper pass)
//   Big  [2][NT][S/4]     the S-wide column tiles of the group update
//   Gs, ds                floats: the head's G and dt of the chunk (256 each)
// kG lanes share a token group, which owns kTok tokens: RT = (256 / kG) kTok.
template <int kS, int kG, int kTok>
struct MainSmem {
  static constexpr int NG = kThreads / kG, RT = NG * kTok, NT = kTT, S4 = kS / 4, P4 = kP / 4;
  static constexpr int KU = RT + 4, KL = NT + 4, WR = 256 + 4, CB = kG / kTok;
  static constexpr int KT4 = (NT * KU > RT * KL ? NT * KU : RT * KL) / 4;
  static constexpr int Wsum = 0, U2 = Wsum + RT * WR / 4, Kt = U2 + 2 * NT * P4,
                       Wt = Kt + 2 * KT4, Qp = Wt + RT * KL / 4, Big = Qp + RT * CB / 4,
                       end4 = Big + 2 * NT * S4;
  static constexpr size_t bytes = 16 * (size_t)end4 + 2 * 256 * sizeof(float);
  static constexpr int kCtas = bytes <= 113 * 1024 ? 2 : 1;  // CTAs per SM
  static_assert(RT % kTT == 0 && RT <= 2 * kTT, "row tiles of 32 or 64 tokens");
  static_assert(S4 % kG == 0 && P4 % kG == 0, "whole float4 slots per lane");
  static_assert(CB >= 1 && NT % CB == 0 && (RT * CB) % 4 == 0, "columns per reduce-scatter");
};

// One CTA per (row tile of RT tokens of a chunk, chunk, batch * group), 256
// threads: thread = (token group grp = tid / kG, lane lg = tid % kG), the
// group owning tokens grp + NG r (r < kTok) of the tile and lane lg the
// float4 slots kG i + lg of every feature row.  Two passes over the chunk's
// 32-token column tiles:
//   upper (columns s >= t): dx_t += dt_t w (B_t . C_s) gy_s,
//                           dB_t += sum_h dt_t w (x_t . gy_s) C_s,  w = exp2(G_s - G_t);
//   lower (columns j <= t): ysm_t += w (C_t . B_j) x_j,
//                           dC_t += sum_h w (gy_t . x_j) B_j,  w = exp2(G_t - G_j) dt_j.
// In each pass the CTA walks the group's heads: per head the P-wide part
// (the scores x . gy or gy . x, dx or ysm, their state terms, the per-token
// scalars), while the S-side weights dt_t w (x . gy) or w (gy . x) are
// added up over the heads in Wsum; the S-wide update then runs once per
// group, B and C being shared by its heads, and writes dB or dC.  c_t . B_j
// comes from the Kcb GEMM, and the state terms from the GEMMs around this
// kernel: dx += dt_t exp2(G_last - G_t) (R B_t) and ysm += exp2(G_t) (h c_t)
// from dxS and ysmS computed before it; dB and dC get R^T x~ and h^T gy~
// added after it.
template <int kS, int kG, int kTok>
__global__ void __launch_bounds__(kThreads, MainSmem<kS, kG, kTok>::kCtas)
bwd_main_kernel(const float *__restrict__ x, const float *__restrict__ dt,
                const float *__restrict__ Bm, const float *__restrict__ Cm,
                const float *__restrict__ D, const float *__restrict__ gy,
                const float *__restrict__ G, const float *__restrict__ dxS,
                const float *__restrict__ ysmS, const float *__restrict__ Kcb,
                float *__restrict__ dx, float *__restrict__ dB, float *__restrict__ dC,
                float *__restrict__ qB, float *__restrict__ dG, float *__restrict__ gyx, int *err,
                int L, int nh, int hpg, int T, int nc, int nb, int nslice) {
  using SM = MainSmem<kS, kG, kTok>;
  constexpr int NG = SM::NG, RT = SM::RT, NT = SM::NT, S4 = SM::S4, P4 = SM::P4;
  constexpr int KU = SM::KU, KL = SM::KL, WR = SM::WR, CB = SM::CB, KTF = 4 * SM::KT4;
  constexpr int QS = S4 / kG, QP = P4 / kG;
  extern __shared__ float4 sm4[];
  float *Wsum = reinterpret_cast<float *>(sm4 + SM::Wsum);
  float4 *U2 = sm4 + SM::U2, *Big = sm4 + SM::Big;
  float *Kt = reinterpret_cast<float *>(sm4 + SM::Kt);
  float *Wt = reinterpret_cast<float *>(sm4 + SM::Wt);
  float *Qp = reinterpret_cast<float *>(sm4 + SM::Qp);
  float *Gs = reinterpret_cast<float *>(sm4 + SM::end4);
  float *ds = Gs + 256;
  const int ntile = T / RT, ng = nh / hpg;
  const int k = blockIdx.x / ntile, tau = blockIdx.x - k * ntile;
  // blockIdx.y = (batch * group) * nslice + slice: the slice's heads are
  // hps consecutive heads of the group; with several slices dB and dC are
  // this slice's share, slice-major (summed by bwd_reduce_kernel)
  const int sl = blockIdx.y % nslice, bg = blockIdx.y / nslice, b = bg / ng, g = bg - b * ng;
  const int hps = hpg / nslice;
  const int tok0 = k * T, valid = min(T, L - tok0);
  const int tid = threadIdx.x, grp = tid / kG, lg = tid % kG, lane = tid & 31;
  // extents (elements per row width) of the buffers, for the debug-bounds checks
  const int64_t ext_h = (int64_t)nb * L * nh, ext_g = (int64_t)nb * L * ng;
  (void)ext_h, (void)ext_g;  // read by the debug-bounds checks only
  // every chunk-indexed buffer of this (chunk, group) and of its heads:
  // checked once, uniform over the CTA
  if (!SSD_IN_BOUNDS(b < nb && k < nc && (int64_t)bg * nc + k < (int64_t)nb * ng * nc, err, 201))
    return;
  if (tau * RT >= valid) return;  // tile past the sequence
  int t[kTok];
  bool live[kTok];
#pragma unroll
  for (int r = 0; r < kTok; ++r) {
    t[r] = tau * RT + NG * r + grp;
    live[r] = t[r] < valid;
  }
  const int64_t tokrow0 = (int64_t)b * L + tok0;  // token row of the chunk's token 0
  const int64_t rowg0 = tokrow0 * ng + g;
  const float *Kc = Kcb + ((int64_t)bg * nc + k) * T * T;
  // stage `rows` tokens from chunk-relative token t0 of a tensor of rows
  // row0 + tok * rstride and width 4 W4 floats, zeros past the sequence
  auto stage = [&](float4 *dst, const float *src, int64_t row0, int rstride, int W4, int t0,
                   int rows, int64_t ext) {
    for (int e = tid; e < rows * W4; e += kThreads) {
      const int r = e / W4, c = e - r * W4, tok = t0 + r;
      const int64_t si = (row0 + (int64_t)(tok < valid ? tok : 0) * rstride) * (4 * W4) + 4 * c;
      const bool ok = tok < valid && SSD_IN_BOUNDS(si + 4 <= ext * 4 * W4, err, 206);
      cp_async16(dst + e, ok ? src + si : src, ok);
    }
  };
  // one pass: kUp = the upper one (dx, dB) or the lower one (ysm, dC)
  auto pass = [&](auto up_c) {
    constexpr bool kUp = decltype(up_c)::value;
    const float *own_h = kUp ? x : gy;    // a head's own rows (x or gy)
    const float *col_h = kUp ? gy : x;    // a head's P-wide column rows
    const float *col_g = kUp ? Cm : Bm;   // the S-wide column rows of the group update
    const int ucount = (valid + NT - 1) / NT;
    const int u0 = kUp ? tau * RT / NT : 0;
    const int u1 = kUp ? ucount : min(ucount, (tau + 1) * RT / NT);
    __syncthreads();  // the previous pass is done with every buffer
    for (int e = tid; e < RT * WR; e += kThreads) Wsum[e] = 0.f;
    cp_async_commit();
    float4 accS[kTok][QS];
#pragma unroll
    for (int r = 0; r < kTok; ++r)
#pragma unroll
      for (int i = 0; i < QS; ++i) accS[r][i] = make_float4(0.f, 0.f, 0.f, 0.f);
    // stage the c . B values of column tile u and the row tile into buffer
    // buf: upper Kt[j][rr] = c_s . B_t, lower Kt[rr][j] = c_t . B_j
    auto stage_k = [&](int buf, int u) {
      float *dst = Kt + buf * KTF;
      constexpr int rows = kUp ? NT : RT, cols4 = (kUp ? RT : NT) / 4;
      for (int e = tid; e < rows * cols4; e += kThreads) {
        const int r = e / cols4, c4 = e - r * cols4;
        const int i = kUp ? u * NT + r : tau * RT + r;
        const int j = kUp ? tau * RT + 4 * c4 : u * NT + 4 * c4;
        cp_async16(dst + r * (kUp ? KU : KL) + 4 * c4, Kc + (int64_t)i * T + j, true);
      }
    };
    for (int hi = sl * hps; hi < (sl + 1) * hps; ++hi) {
      const int h = g * hpg + hi;
      const int64_t rowh0 = tokrow0 * nh + h, bh = (int64_t)b * nh + h;
      __syncthreads();  // the previous head is done with Gs, ds, U2, Kt, Wt, Qp and Big
      const float *Gc = G + (bh * nc + k) * T;
      for (int i = tid; i < T; i += kThreads) {
        Gs[i] = Gc[i];
        const int64_t di = rowh0 + (int64_t)i * nh;
        ds[i] = i < valid && SSD_IN_BOUNDS(di < ext_h, err, 209) ? dt[di] : 0.f;
      }
      // this head's own rows x_t (upper) or gy_t (lower), this lane's slots
      float4 rP[kTok][QP], accP[kTok][QP];
#pragma unroll
      for (int r = 0; r < kTok; ++r)
#pragma unroll
        for (int i = 0; i < QP; ++i) {
          const int64_t hi4 = (rowh0 + (int64_t)t[r] * nh) * kP + 4 * (kG * i + lg);
          rP[r][i] = live[r] && SSD_IN_BOUNDS(hi4 + 4 <= ext_h * kP, err, 208)
                         ? *reinterpret_cast<const float4 *>(own_h + hi4)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
          accP[r][i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      float qacc = 0.f;  // this lane's share of q . B for its token of the scatter
      int r_own = 0, c_own = 0;
      stage(U2, col_h, rowh0, nh, P4, u0 * NT, NT, ext_h);
      stage_k(0, u0);
      cp_async_commit();
      __syncthreads();  // Gs and ds
      float Gt[kTok], dtt[kTok];
#pragma unroll
      for (int r = 0; r < kTok; ++r) {
        Gt[r] = Gs[t[r]];
        dtt[r] = ds[t[r]];
      }
      for (int u = u0; u < u1; ++u) {
        const int cur = (u - u0) & 1;
        if (u + 1 < u1) {
          stage(U2 + (cur ^ 1) * NT * P4, col_h, rowh0, nh, P4, (u + 1) * NT, NT, ext_h);
          stage_k(cur ^ 1, u + 1);
        }
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const float4 *u2p = U2 + cur * NT * P4 + lg;
        const float *ktp = Kt + cur * KTF;
        // token r meets this column tile at all unless its 32-token block
        // lies wholly on the masked side of the diagonal; the loop body is
        // compiled once per set of active blocks (uniform over the CTA, so
        // the shuffles stay warp-wide)
        auto tile = [&](auto mask_c) {
          constexpr int kMask = decltype(mask_c)::value;
          auto on = [](int r) { return ((kMask >> ((r * NG) / kTT)) & 1) != 0; };
          // scores x_t . gy_s (upper) or gy_t . x_j (lower) of the group's
          // tokens, CB columns at a time, summed over the group's lanes by one
          // reduce-scatter (one total per lane), turned by that lane into the
          // pair's P-side weight (Wt) and its S-side one (added to Wsum)
#pragma unroll 2
          for (int j0 = 0; j0 < NT; j0 += CB) {
            float v[kG];
#pragma unroll
            for (int c = 0; c < CB; ++c) {
              float4 cP[QP];
#pragma unroll
              for (int i = 0; i < QP; ++i) cP[i] = u2p[(j0 + c) * P4 + kG * i];
#pragma unroll
              for (int r = 0; r < kTok; ++r) {
                float a = 0.f;
                if (on(r)) {
#pragma unroll
                  for (int i = 0; i < QP; ++i) a = dot4(rP[r][i], cP[i], a);
                }
                v[c * kTok + r] = a;
              }
            }
            int idx;
            const float d = group_scatter<kG>(v, lane, &idx);
            r_own = idx % kTok;
            c_own = idx / kTok;
            const int j = j0 + c_own, s = u * NT + j;
            const int rr = NG * r_own + grp, tr = tau * RT + rr;
            const float Gc2 = Gs[s], Gr = Gs[tr];
            float w = 0.f;
            if (kUp) {
              if (s >= tr && s < valid && tr < valid) w = exp2f(Gc2 - Gr);
            } else {
              if (s <= tr && tr < valid) w = exp2f(Gr - Gc2) * ds[s];  // dt = 0 past the sequence
            }
            const float cb = kUp ? ktp[j * KU + rr] : ktp[rr * KL + j];
            const float dtr = kUp ? ds[tr] : 1.f;
            Wt[rr * KL + j] = dtr * w * cb;
            Wsum[rr * WR + s] += dtr * w * d;
            if (kUp) qacc = fmaf(w * d, cb, qacc);
          }
          __syncwarp();  // a group's weights come from its own lanes
          // the P-wide update: every column row loaded serves the group's tokens
#pragma unroll 4
          for (int j = 0; j < NT; ++j) {
            float4 cP[QP];
#pragma unroll
            for (int i = 0; i < QP; ++i) cP[i] = u2p[j * P4 + kG * i];
#pragma unroll
            for (int r = 0; r < kTok; ++r) {
              if (!on(r)) continue;
              const float aP = Wt[(NG * r + grp) * KL + j];
#pragma unroll
              for (int i = 0; i < QP; ++i) axpy4(aP, cP[i], accP[r][i]);
            }
          }
          __syncwarp();  // the weights are rewritten for the next tile
        };
        int mask = 0;
#pragma unroll
        for (int rb = 0; rb < RT / kTT; ++rb)
          if (kUp ? u * NT + NT > tau * RT + kTT * rb : u * NT < tau * RT + kTT * rb + kTT)
            mask |= 1 << rb;
        if (RT == kTT || mask == 3)
          tile(std::integral_constant<int, 3>{});
        else if (mask == 1)
          tile(std::integral_constant<int, 1>{});
        else
          tile(std::integral_constant<int, 2>{});
        __syncthreads();  // tile u's buffers are refilled two iterations on
      }
      cp_async_wait<0>();
      // the state term of this head's tokens, formed by the GEMMs before
      // this kernel: raw = R_k B_t (upper) or h_k c_t (lower), this lane's
      // P slots; dx += dt_t exp2(G_last - G_t) raw, ysm += exp2(G_t) raw
      const float GL = Gs[valid - 1];
      const float *stP = kUp ? dxS : ysmS;
      float qst[kTok];  // x_t . (R B_t), this lane's slots (upper)
#pragma unroll
      for (int r = 0; r < kTok; ++r) {
        const float f = live[r] ? (kUp ? dtt[r] * exp2f(GL - Gt[r]) : exp2f(Gt[r])) : 0.f;
        qst[r] = 0.f;
#pragma unroll
        for (int i = 0; i < QP; ++i) {
          const int64_t si = (rowh0 + (int64_t)t[r] * nh) * kP + 4 * (kG * i + lg);
          const float4 raw = live[r] && SSD_IN_BOUNDS(si + 4 <= ext_h * kP, err, 207)
                                 ? *reinterpret_cast<const float4 *>(stP + si)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
          if (kUp) qst[r] = dot4(rP[r][i], raw, qst[r]);
          axpy4(f, raw, accP[r][i]);
        }
      }
      // the head's per-token outputs
      if (kUp) {
        Qp[(NG * r_own + grp) * CB + c_own] = qacc;  // this lane's share, one slot each
        const float Dh = D ? D[h] : 0.f;
#pragma unroll
        for (int r = 0; r < kTok; ++r) {
          float v3[4] = {0.f, qst[r], 0.f, 0.f};  // x . (dx - D gy), x . R B, x . gy
          const int64_t rh = rowh0 + (int64_t)t[r] * nh;
#pragma unroll
          for (int i = 0; i < QP; ++i) {
            const int f = 4 * (kG * i + lg);
            const bool ok = live[r] && SSD_IN_BOUNDS(rh * kP + f + 4 <= ext_h * kP, err, 210);
            const float4 gq = ok ? *reinterpret_cast<const float4 *>(gy + rh * kP + f)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            v3[0] = dot4(rP[r][i], accP[r][i], v3[0]);
            v3[2] = dot4(rP[r][i], gq, v3[2]);
            if (ok) {
              float4 o = accP[r][i];
              axpy4(Dh, gq, o);
              *reinterpret_cast<float4 *>(dx + rh * kP + f) = o;
            }
          }
          group_sums<4, kG>(v3, lane);
          __syncwarp();  // the group's shares of q . B are in Qp
          if (lg == 0 && live[r]) {
            const int rr = NG * r + grp;
            float q = (kUp ? exp2f(GL - Gt[r]) : 0.f) * v3[1];
#pragma unroll
            for (int c = 0; c < CB; ++c) q += Qp[rr * CB + c];
            const int64_t o = (bh * nc + k) * T + t[r];
            qB[o] = q;
            dG[o] = -v3[0];
            gyx[o] = v3[2];
          }
        }
      } else {
#pragma unroll
        for (int r = 0; r < kTok; ++r) {
          float gd[1] = {0.f};
#pragma unroll
          for (int i = 0; i < QP; ++i) gd[0] = dot4(rP[r][i], accP[r][i], gd[0]);  // gy . ysm
          group_sums<1, kG>(gd, lane);
          if (lg == 0 && live[r]) {
            const int64_t o = (bh * nc + k) * T + t[r];
            dG[o] += gd[0];  // the upper pass of this thread stored -x . dxsm
          }
        }
      }
    }
    // the group update: accS[s] += sum_s' Wsum[t][s'] col_s' over the pass's
    // columns, S-wide column tiles double-buffered in Big
    __syncthreads();  // Wsum complete, Big free
    stage(Big, col_g, rowg0, ng, S4, u0 * NT, NT, ext_g);
    cp_async_commit();
    for (int u = u0; u < u1; ++u) {
      const int cur = (u - u0) & 1;
      if (u + 1 < u1) stage(Big + (cur ^ 1) * NT * S4, col_g, rowg0, ng, S4, (u + 1) * NT, NT, ext_g);
      cp_async_commit();
      cp_async_wait<1>();
      __syncthreads();
      const float4 *u1p = Big + cur * NT * S4 + lg;
#pragma unroll 2
      for (int j = 0; j < NT; ++j) {
        float4 cS[QS];
#pragma unroll
        for (int i = 0; i < QS; ++i) cS[i] = u1p[j * S4 + kG * i];
#pragma unroll
        for (int r = 0; r < kTok; ++r) {
          const float a = Wsum[(NG * r + grp) * WR + u * NT + j];
#pragma unroll
          for (int i = 0; i < QS; ++i) axpy4(a, cS[i], accS[r][i]);
        }
      }
      __syncthreads();
    }
    cp_async_wait<0>();
    float *out = (kUp ? dB : dC) + (int64_t)sl * ext_g * kS;
#pragma unroll
    for (int r = 0; r < kTok; ++r) {
      if (!live[r]) continue;
      const int64_t rg = (rowg0 + (int64_t)t[r] * ng) * kS;
#pragma unroll
      for (int i = 0; i < QS; ++i)
        if (SSD_IN_BOUNDS(rg + 4 * (kG * i + lg) + 4 <= ext_g * kS, err, 212))
          *reinterpret_cast<float4 *>(out + rg + 4 * (kG * i + lg)) = accS[r][i];
    }
  };
  pass(std::integral_constant<bool, true>{});
  pass(std::integral_constant<bool, false>{});
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
  // every chunk-indexed buffer of this (chunk, head) (R, states, qB, dG,
  // gyx, part) and its final state: checked once, uniform over the CTA
  if (!SSD_IN_BOUNDS(b < nb && k < nc && h < nh && (int64_t)bh * nc + k < (int64_t)nb * nh * nc,
                     err, 202))
    return;
  // <R_k, h_{k+1}> over P x S
  // R and the states are chunk-major, [b, nc, nh, P, S]
  const float *Rk = R + (((int64_t)b * nc + k) * nh + h) * P * S;
  const float *hn = k + 1 < nc ? states + (((int64_t)b * nc + k + 1) * nh + h) * P * S
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
    const int64_t di = ((int64_t)b * L + tok0 + tid) * nh + h;
    const bool ok = SSD_IN_BOUNDS(di < (int64_t)nb * L * nh, err, 213);
    const float dtt = ok ? dt[di] : 0.f;
    if (ok) ddt[di] = A[h] * eta + qB[o];
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

// dB and dC, the sums of the head slices' shares (slice-major, nslice > 1)
// in slice order, one thread per element; then (threads past those) dA and
// dD per head, the sums of the per-chunk shares over batches and chunks in a
// fixed order.
__global__ void __launch_bounds__(kThreads)
bwd_reduce_kernel(const float *__restrict__ sB, const float *__restrict__ sC,
                  float *__restrict__ dB, float *__restrict__ dC, int64_t n_bc, int nslice,
                  const float2 *__restrict__ part, float *__restrict__ dA, float *__restrict__ dD,
                  int nh, int nc, int nb, int *err) {
  const int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  if (e < n_bc) {
    float sb = 0.f, sc = 0.f;
    for (int i = 0; i < nslice; ++i) {
      sb += sB[i * n_bc + e];
      sc += sC[i * n_bc + e];
    }
    dB[e] = sb;
    dC[e] = sc;
    return;
  }
  if (e - n_bc >= nh) return;
  const int h = (int)(e - n_bc);
  float a = 0.f, d = 0.f;
  for (int b = 0; b < nb; ++b)
    for (int k = 0; k < nc; ++k) {
      const int64_t pi = ((int64_t)b * nh + h) * nc + k;
      if (!SSD_IN_BOUNDS(pi < (int64_t)nb * nh * nc, err, 215)) continue;
      const float2 v = part[pi];
      a += v.x;
      d += v.y;
    }
  dA[h] = a;
  if (dD) dD[h] = d;
}

// ------------------------------------------------------------ bf16 <-> fp32

// The bf16 I/O of ssd_backward: up to five tensors converted in one launch
// (bf16 -> fp32 before the fp32 pass, fp32 -> bf16 of its outputs after
// it), eight elements a step where a segment allows (16-byte aligned
// pointers, as the library requires), the tail one by one.
__global__ void __launch_bounds__(kThreads)
bwd_convert_kernel(const BwdConvert a) {
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  const int64_t first = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  for (int sg = 0; sg < a.nseg; ++sg) {
    const int64_t n = a.seg[sg].n, n8 = n / 8;
    if (a.to_bf16) {
      const float4 *src = static_cast<const float4 *>(a.seg[sg].src);
      uint4 *dst = static_cast<uint4 *>(a.seg[sg].dst);
      for (int64_t i = first; i < n8; i += stride) {
        const float4 lo = src[2 * i], hi = src[2 * i + 1];
        __nv_bfloat162 o[4] = {__floats2bfloat162_rn(lo.x, lo.y), __floats2bfloat162_rn(lo.z, lo.w),
                               __floats2bfloat162_rn(hi.x, hi.y), __floats2bfloat162_rn(hi.z, hi.w)};
        dst[i] = *reinterpret_cast<const uint4 *>(o);
      }
      const float *s1 = static_cast<const float *>(a.seg[sg].src);
      __nv_bfloat16 *d1 = static_cast<__nv_bfloat16 *>(a.seg[sg].dst);
      for (int64_t i = 8 * n8 + first; i < n; i += stride) d1[i] = __float2bfloat16_rn(s1[i]);
    } else {
      const uint4 *src = static_cast<const uint4 *>(a.seg[sg].src);
      float4 *dst = static_cast<float4 *>(a.seg[sg].dst);
      for (int64_t i = first; i < n8; i += stride) {
        const uint4 v = src[i];
        const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&v);
        const float2 f0 = __bfloat1622float2(b2[0]), f1 = __bfloat1622float2(b2[1]),
                     f2 = __bfloat1622float2(b2[2]), f3 = __bfloat1622float2(b2[3]);
        dst[2 * i] = make_float4(f0.x, f0.y, f1.x, f1.y);
        dst[2 * i + 1] = make_float4(f2.x, f2.y, f3.x, f3.y);
      }
      const __nv_bfloat16 *s1 = static_cast<const __nv_bfloat16 *>(a.seg[sg].src);
      float *d1 = static_cast<float *>(a.seg[sg].dst);
      for (int64_t i = 8 * n8 + first; i < n; i += stride) d1[i] = __bfloat162float(s1[i]);
    }
  }
}

}  // namespace

cudaError_t launch_bwd_convert(const BwdConvert &a, cudaStream_t st) {
  int64_t n = 0;
  for (int i = 0; i < a.nseg; ++i) n = std::max<int64_t>(n, a.seg[i].n);
  const int64_t want = (n / 8 + kThreads - 1) / kThreads;
  const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>(want, 4 * (int64_t)sm_count()));
  bwd_convert_kernel<<<blocks, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

bool bwd_supported(const Dims &d) {
  // chunks of whole row tiles of the per-token kernel: 64 tokens at dstate
  // 256, 32 below
  const int64_t rt = d.S == 256 ? 2 * kTT : kTT;
  return d.P == kP && (d.S == 64 || d.S == 128 || d.S == 256) && d.T >= rt && d.T % rt == 0 &&
         d.T <= 256 && bwd_state_gemm_supported(d);
}

int bwd_head_slices(const Dims &d) {
  // 64-token row tiles, one CTA per SM, at dstate 256; 32-token tiles, two
  // CTAs per SM, below: slice the heads of a group until the grid fills two
  // waves of a 152-SM GB300 (the fewest slices that do; a divisor of the
  // heads per group, at most 8)
  const int64_t rt = d.S == 256 ? 64 : 32, per_sm = d.S == 256 ? 1 : 2;
  const int64_t base = d.b * d.ng * d.nc * (d.T / rt), want = 2 * 152 * per_sm;
  int best = 1;
  for (int n = 1; n <= 8 && n <= d.hpg; ++n)
    if (d.hpg % n == 0) {
      best = n;
      if (base * n >= want) break;
    }
  return best;
}



namespace {
template <int kS, int kG, int kTok>
cudaError_t launch_main(const Dims &d, const float *x, const float *dt, const float *B,
                        const float *C, const float *D, const float *gy, const float *G,
                        const float *dxS, const float *ysmS, const float *Kcb, float *dx,
                        float *dB, float *dC, float *qB, float *dG, float *gyx, int *err,
                        cudaStream_t st) {
  using SM = MainSmem<kS, kG, kTok>;
  const size_t smem = SM::bytes;
  cudaError_t e = cudaFuncSetAttribute(bwd_main_kernel<kS, kG, kTok>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int nslice = bwd_head_slices(d);
  dim3 grid((unsigned)(d.nc * (d.T / SM::RT)), (unsigned)(d.b * d.ng * nslice));
  bwd_main_kernel<kS, kG, kTok><<<grid, kThreads, smem, st>>>(
      x, dt, B, C, D, gy, G, dxS, ysmS, Kcb, dx, dB, dC, qB, dG, gyx, err, (int)d.L,
      (int)d.nh, (int)d.hpg, (int)d.T, (int)d.nc, (int)d.b, nslice);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_bwd_main(const Dims &d, const float *x, const float *dt, const float *B,
                            const float *C, const float *D, const float *gy, const float *G,
                            const float *dxS, const float *ysmS, const float *Kcb, float *dx,
                            float *dB, float *dC, float *qB, float *dG, float *gyx, int *err,
                            cudaStream_t st) {
  // 16-lane token groups: four tokens (64-token row tiles, one CTA per SM)
  // at dstate 256, two (32-token tiles, two CTAs per SM) below, measured at
  // b1 L32768 h48 g8 (S 256) and b2 L16384 h32 (S 64, 128): 15.9 ms at S =
  // 256; 6.97 / 5.74 ms at S = 128 / 64 against 7.43 / 6.57 with four tokens
  // and one CTA
  switch (d.S) {
    case 64:
      return launch_main<64, 16, 2>(d, x, dt, B, C, D, gy, G, dxS, ysmS, Kcb, dx, dB, dC, qB,
                                    dG, gyx, err, st);
    case 128:
      return launch_main<128, 16, 2>(d, x, dt, B, C, D, gy, G, dxS, ysmS, Kcb, dx, dB, dC, qB,
                                     dG, gyx, err, st);
    default:
      return launch_main<256, 16, 4>(d, x, dt, B, C, D, gy, G, dxS, ysmS, Kcb, dx, dB, dC, qB,
                                     dG, gyx, err, st);
  }
}

cudaError_t launch_bwd_scale(const Dims &d, const float *x, const float *gy, const float *dt,
                             const float *G, float *xs, float *gys, int *err, cudaStream_t st) {
  const int64_t n4 = d.b * d.L * d.nh * (kP / 4);
  const int blocks = (int)std::max<int64_t>(
      1, std::min<int64_t>((n4 + kThreads - 1) / kThreads, 8 * (int64_t)sm_count()));
  bwd_scale_kernel<<<blocks, kThreads, 0, st>>>(x, gy, dt, G, xs, gys, err, (int)d.L, (int)d.nh,
                                                (int)d.T, (int)d.nc, (int)d.b);
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

cudaError_t launch_bwd_reduce(const Dims &d, const float *sB, const float *sC, float *dB,
                              float *dC, const float2 *part, float *dA, float *dD, int *err,
                              cudaStream_t st) {
  const int nslice = bwd_head_slices(d);
  const int64_t n_bc = nslice > 1 ? d.b * d.L * d.ng * d.S : 0;
  const int64_t n = n_bc + d.nh;
  bwd_reduce_kernel<<<(unsigned)((n + kThreads - 1) / kThreads), kThreads, 0, st>>>(
      sB, sC, dB, dC, n_bc, nslice, part, dA, dD, (int)d.nh, (int)d.nc, (int)d.b, err);
  return cudaGetLastError();
}

}  // namespace ssd
