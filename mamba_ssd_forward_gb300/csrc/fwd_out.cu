// Forward path, output pass (bf16 I/O) with the decay factored about one
// anchor per chunk and head, so that the masked interaction tile C B^T of a
// chunk is the A operand of every head of its group unchanged.
//
// The page's chunked output equation ("Accelerating Mamba-2 with
// High-Performance Forward Pass Kernels in NVIDIA CUDA Tile", section
// "Mamba-2 architecture", the compute_out step):
//
//   y_i = exp2(G_i) (h_k c_i) + sum_{j<=i in chunk} (c_i . B_j) exp2(G_i - G_j) dt_j x_j
//         + D x_i
//
// with G the in-chunk cumsum of A dt in log2 units.  For any anchor value
// alpha, exp2(G_i - G_j) = exp2(G_i - alpha) exp2(alpha - G_j) and
// exp2(G_i) = exp2(G_i - alpha) exp2(alpha), so
//
//   y_i = u_i [ c_i . (2^alpha h_k) + sum_{j<=i} (c_i . B_j) xh_j ] + D x_i,
//   u_i = exp2(G_i - alpha),   xh_j = exp2(alpha - G_j) dt_j x_j.
//
// The bracket is one accumulation: C (2^alpha h)^T plus (C B^T masked) Xh.
// The masked C B^T carries no decay, so it is computed and rounded to bf16
// once per chunk and shared by the heads of the group; per head the row
// warps only scale each x row by its factor and apply u_i in the epilogue.
// alpha is the integer nearest half the chunk's total decay (so 2^alpha h
// is exact in bf16, and every factor stays within 2^+-(span / 2): the
// method's own rule of never keeping positive exponents holds for the
// product u_i xh_j, exponent G_i - G_j <= 0, while each factor stays
// bounded).  The chunk-jump kernel, which forms each chunk's cumsum anyway,
// writes alpha, u and v, and the state pass stores the start states already
// times 2^alpha.  A chunk whose decay is too steep for bounded factors (the
// chunk-jump kernel flags it: total decay above 2^-180, or a real token's
// factor below 2^-120) takes an exact per-element path here instead: its
// state is stored unscaled, and the epilogue forms exp2(G_i - G_j) dt_j per
// pair on the CUDA cores from the packed C B^T and the raw x rows (slow but
// exact; such chunks are rare).
//
// One CTA per (slice of hs heads of one group, chunk, batch):
//   producer warp: C of the chunk (resident), then through a ring of 16 KB
//     stages: phase 1's B blocks (128 tokens x 64 of S), then per head its
//     start state (128 rows of S x 64 p per stage) and its x rows (128
//     tokens x 64 p per stage);
//   MMA warp: phase 1 C B^T into tensor memory in fp32 (row tile t of the
//     chunk x token block of B); then per head into one of two accumulator
//     sets: Acc_t = C_t (2^alpha h)^T, then + (C B^T)_t Xh with the packed
//     masked tile read from tensor memory as the A operand;
//   row warps (8): pack C B^T in place to masked bf16 pairs; per head the
//     scaling of the x stages (thread = row) and the epilogue
//     y = u_i Acc_i + D x_i, staged in a y buffer of its own and stored by
//     TMA (so an x stage is free as soon as the MMAs that read it are done,
//     and the ring never waits on an epilogue).  Stage barriers take one
//     arrival per warp.
// Supported: P = 64, S a multiple of 64 up to 256, T in {128, 256}.
#include "fwd.cuh"

namespace ssd {
namespace {

constexpr int kRowWarps = 8;
constexpr int kRowThreads = kRowWarps * 32;
constexpr int kThreads = kRowThreads + 64;
constexpr int kProducerWarp = kRowWarps, kMmaWarp = kRowWarps + 1;
constexpr int kP = 64;
constexpr int kStage = 128 * 128;  // one ring stage: 128 rows of 128 bytes
constexpr int kMaxSlots = 8;

struct OutArgs {
  const __nv_bfloat16 *dt;
  const float *A, *D;
  // per-token factors u, v [b, nh, nc * T] and per-chunk anchors [b, nh,
  // nc] = (alpha, steep ? 1 : 0), from the chunk-jump kernel
  const float *u, *v;
  const float2 *anchor;
  int *err;
  int L, nh, S, hpg, T, nc, hs, nslot, nyst;
  int nb;  // batch count (the extents the debug-bounds checks use)
};

__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&b);
}

// Tensor-memory columns.  T = 256: phase 1 C B^T fp32, row tile 1 at [0,
// 256) and row tile 0 at [256, 384), packed in place to bf16 pairs at [0,
// 128) and [256, 320); accumulator set 0 at [128, 256), set 1 at [320,
// 448), row tile t at +64 t.  T = 128: C B^T fp32 at [0, 128), packed to
// [0, 64); accumulator sets at 128 and 192.
template <int kT>
struct Cols {
  static __device__ __forceinline__ uint32_t scf(int t) {
    return kT == 256 ? (t ? 0u : 256u) : 0u;
  }
  static __device__ __forceinline__ uint32_t pk(int t) { return scf(t); }
  static __device__ __forceinline__ uint32_t acc(int set, int t) {
    return kT == 256 ? (set ? 320u : 128u) + 64u * (uint32_t)t : 128u + 64u * (uint32_t)set;
  }
  static constexpr uint32_t kAlloc = kT == 256 ? 512u : 256u;
};

template <int kT>
__global__ void __launch_bounds__(kThreads, 1)
fwd_out_bf16(const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_B,
             const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_st,
             const __grid_constant__ CUtensorMap tm_y, const OutArgs a) {
  using TC = Cols<kT>;
  constexpr int nT = kT / 128;  // row tiles of the chunk (and x stages per head)
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  // full: a B or state stage has landed (the MMA warp waits); xfull: an x
  // stage has landed (the row warps wait; they skip the other stages, so
  // their barrier must count x stages only); scaled: the row warps are done
  // with an x stage; empty: the stage's readers are done
  __shared__ __align__(8) uint64_t c_full, full[kMaxSlots], xfull[kMaxSlots], scaled[kMaxSlots],
      empty[kMaxSlots], sc_done, pack_done, acc_full[2], acc_free[2];
  __shared__ uint32_t tmem_slot;
  // a steep head's G (log2 units) and dt of every token, by head parity
  __shared__ __align__(16) float Gs[2][256];
  __shared__ __align__(16) float dts[2][256];
  __shared__ float warp_tot[kRowWarps];

  const int L = a.L, nh = a.nh, S = a.S, hs = a.hs, nslot = a.nslot;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int k = blockIdx.y, b = blockIdx.z;
  const int hbase = blockIdx.x * hs, g = hbase / a.hpg;
  const int tok0 = k * kT;
  const int valid = min(kT, L - tok0);
  const int nS = S / 64;               // 64-wide blocks of S
  const int nH = (S + 127) / 128;      // state stages per head
  const int hrows = S < 128 ? S : 128; // rows of S in one state stage
  uint8_t *Cs = smem;                  // C tile t, S block sb at (t nS + sb) kStage
  uint8_t *ring = smem + nT * nS * kStage;
  auto slot_ptr = [&](int u) { return ring + (u % nslot) * kStage; };
  // y staging: one 128-row tile per row tile of the chunk, or (a.nyst = 1)
  // one tile that the row tiles take in turn
  uint8_t *ystage = ring + nslot * kStage;

  if (tid == 0) {
    ptx::mbar_init(&c_full, 1);
    for (int i = 0; i < nslot; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&xfull[i], 1);
      ptx::mbar_init(&scaled[i], kRowWarps);  // one arrival per row warp
      ptx::mbar_init(&empty[i], 1);
    }
    ptx::mbar_init(&sc_done, 1);
    ptx::mbar_init(&pack_done, kRowWarps);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&acc_full[i], 1);
      ptx::mbar_init(&acc_free[i], kRowWarps);
    }
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(&tmem_slot, TC::kAlloc);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const bool leader = (tid & 31) == 0;
  const int n_p1 = nS * nT;  // phase-1 stages

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (leader) {
      ptx::prefetch_tmap(&tm_C);
      ptx::prefetch_tmap(&tm_B);
      ptx::prefetch_tmap(&tm_x);
      ptx::prefetch_tmap(&tm_st);
      ptx::mbar_arrive_expect_tx(&c_full, nT * nS * kStage);
      for (int t = 0; t < nT; ++t)
        for (int sb = 0; sb < nS; ++sb)
          ptx::tma_load_4d(Cs + (t * nS + sb) * kStage, &tm_C, sb * 64, g, tok0 + t * 128, b,
                           &c_full);
    }
    __syncwarp();
    int u = 0;
    auto acquire = [&](int code) {
      ptx::mbar_wait(&empty[u % nslot], ((u / nslot) & 1) ^ 1, a.err, code);
    };
    for (int sb = 0; sb < nS; ++sb)
      for (int th = 0; th < nT; ++th, ++u) {
        acquire(140);
        if (leader) {
          ptx::mbar_arrive_expect_tx(&full[u % nslot], kStage);
          ptx::tma_load_4d(slot_ptr(u), &tm_B, sb * 64, g, tok0 + th * 128, b, &full[u % nslot]);
        }
        __syncwarp();
      }
    for (int q = 0; q < hs; ++q) {
      const int h = hbase + q;
      const int row = (b * nh + h) * a.nc + k;  // this head's start state
      for (int hh = 0; hh < nH; ++hh, ++u) {
        acquire(141);
        if (leader) {
          // the start states come from the preceding kernel (the state
          // pass), which may still be running when this CTA starts
          if (q == 0 && hh == 0) ptx::griddep_wait();
          ptx::mbar_arrive_expect_tx(&full[u % nslot], hrows * 128);
          ptx::tma_load_3d(slot_ptr(u), &tm_st, 0, hh * 128, row, &full[u % nslot]);
        }
        __syncwarp();
      }
      for (int xt = 0; xt < nT; ++xt, ++u) {
        acquire(142);
        if (leader) {
          ptx::mbar_arrive_expect_tx(&xfull[u % nslot], kStage);
          ptx::tma_load_4d(slot_ptr(u), &tm_x, 0, h, tok0 + xt * 128, b, &xfull[u % nslot]);
        }
        __syncwarp();
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // parity of the next wait on full[slot] / scaled[slot], one bit per slot
    // (each barrier counts only the stages this warp waits on it for)
    uint32_t fpar = 0, spar = 0;
    auto wait_full = [&](int v, int code) {
      const int sl = v % nslot;
      ptx::mbar_wait(&full[sl], (fpar >> sl) & 1, a.err, code);
      fpar ^= 1u << sl;
    };
    ptx::mbar_wait(&c_full, 0, a.err, 143);
    ptx::tc_fence_after();
    int u = 0;
    const uint32_t idCB = ptx::idesc_bf16(128, 128, false, false);
    for (int sb = 0; sb < nS; ++sb)
      for (int th = 0; th < nT; ++th, ++u) {
        wait_full(u, 144);
        ptx::tc_fence_after();
        if (leader) {
          const uint32_t b0 = ptx::smem_u32(slot_ptr(u));
          for (int t = th; t < nT; ++t) {
            const uint32_t c0 = ptx::smem_u32(Cs + (t * nS + sb) * kStage);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t cd = ptx::smem_desc(c0 + kk * 32, 16, 1024, ptx::kSw128);
              const uint64_t bd = ptx::smem_desc(b0 + kk * 32, 16, 1024, ptx::kSw128);
              ptx::mma_ss<false>(tmem + TC::scf(t) + 128 * th, cd, bd, idCB,
                                 (sb | kk) ? 1u : 0u);
            }
          }
          ptx::mma_commit(&empty[u % nslot]);
        }
        __syncwarp();
      }
    if (leader) ptx::mma_commit(&sc_done);
    __syncwarp();
    const uint32_t idY = ptx::idesc_bf16(128, kP, false, true);
    ptx::mbar_wait(&pack_done, 0, a.err, 145);
    ptx::griddep_wait();  // the anchors come from the chunk-jump kernel
    for (int q = 0; q < hs; ++q) {
      const int set = q & 1;
      if (q >= 2) ptx::mbar_wait(&acc_free[set], ((q >> 1) - 1) & 1, a.err, 146);
      ptx::tc_fence_after();
      // the chunk's path, from its anchor
      const int64_t ai = ((int64_t)b * nh + hbase + q) * a.nc + k;
      const int steep = SSD_IN_BOUNDS(ai < (int64_t)a.nb * nh * a.nc, a.err, 61)
                            ? a.anchor[ai].y != 0.f
                            : 0;
      // Acc_t = C_t (2^alpha h)^T over the state stages (stored scaled by the
      // state pass)
      for (int hh = 0; hh < nH; ++hh, ++u) {
        const int sl = u % nslot;
        wait_full(u, 147);
        ptx::tc_fence_after();
        if (leader) {
          const uint32_t h0 = ptx::smem_u32(slot_ptr(u));
          const int nkk = min(128, S - hh * 128) / 16;  // rows of S in this stage / 16
          for (int t = 0; t < nT; ++t)
            for (int kk = 0; kk < nkk; ++kk) {
              const int s16 = hh * 128 + kk * 16;  // first row of S of this K step
              const uint32_t c0 = ptx::smem_u32(Cs + (t * nS + (s16 >> 6)) * kStage);
              const uint64_t cd =
                  ptx::smem_desc(c0 + ((s16 & 63) >> 4) * 32, 16, 1024, ptx::kSw128);
              const uint64_t hd = ptx::smem_desc(h0 + kk * 2048, 8192, 1024, ptx::kSw128);
              ptx::mma_ss<false>(tmem + TC::acc(set, t), cd, hd, idY, (hh | kk) ? 1u : 0u);
            }
          ptx::mma_commit(&empty[sl]);  // the state stage is free once these are done
        }
        __syncwarp();
      }
      // Acc_t += (C B^T)_t Xh over the x stages, each stage free once its
      // MMAs are done (skipped for a steep head, whose epilogue forms the
      // in-chunk sum itself from the raw x stages and then frees them)
      for (int xt = 0; xt < nT; ++xt, ++u) {
        const int sl = u % nslot;
        ptx::mbar_wait(&scaled[sl], (spar >> sl) & 1, a.err, 148);
        spar ^= 1u << sl;
        ptx::tc_fence_after();
        if (leader && !steep) {
          const uint32_t x0 = ptx::smem_u32(slot_ptr(u));
          for (int t = xt; t < nT; ++t)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t xd = ptx::smem_desc(x0 + kk * 2048, 8192, 1024, ptx::kSw128);
              ptx::mma_ts_bf16(tmem + TC::acc(set, t), tmem + TC::pk(t) + 64 * xt + 8 * kk, xd,
                               idY, 1u);
            }
          ptx::mma_commit(&empty[sl]);
        }
        __syncwarp();
      }
      if (leader) ptx::mma_commit(&acc_full[set]);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ row warps
    const int quad = warp & 3;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    // epilogue / x-scaling mapping: T = 256: thread = row tid (row tile
    // tid / 128), all 64 columns; T = 128: row tid % 128, columns
    // 32 (tid / 128) .. +31
    constexpr int kCols = kT == 256 ? 64 : 32;
    const int erow = kT == 256 ? tid : (tid & 127);  // chunk-relative row
    const int etile = erow >> 7;
    const int ecol = kT == 256 ? 0 : 32 * (tid >> 7);
    const int lrow = erow & 127;  // row within its tile = TMEM lane
    const bool tok_ok = tid < valid;

    // one arrival per warp on a barrier, once every lane's writes are done
    auto warp_arrive = [&](uint64_t *bar) {
      __syncwarp();
      if ((tid & 31) == 0) ptx::mbar_arrive(bar);
    };

    // A head's inputs from the chunk-jump kernel and the parameters: this
    // row's factors u and v, the chunk's anchor (alpha, steep) and D,
    // fetched one head ahead so no instruction waits on them.
    struct HeadIn {
      float u, v, D;
      int steep;
    };
    auto fetch_head = [&](int q) {
      HeadIn r;
      const int h = hbase + q;
      const int64_t bhk = ((int64_t)b * nh + h) * a.nc + k;
      const int64_t o = bhk * kT + erow;
      r.u = r.v = r.D = 0.f;
      r.steep = 0;
      if (SSD_IN_BOUNDS(h < nh && bhk < (int64_t)a.nb * nh * a.nc, a.err, 62)) {
        r.u = a.u[o];
        r.v = a.v[o];
        r.steep = a.anchor[bhk].y != 0.f;
        r.D = a.D ? a.D[h] : 0.f;
      }
      return r;
    };

    // ---- phase 1 output: C B^T packed in place to masked bf16 pairs.  The
    // thread of lane r in warps 4 t .. 4 t + 3 packs row r of row tile t
    // (T = 128: warps 0-3 only), reading 32 fp32 columns and writing 16
    // packed ones each step; each step's writes land on columns an earlier
    // step has read.
    ptx::mbar_wait(&sc_done, 0, a.err, 149);
    ptx::tc_fence_after();
    {
      const int pt = warp >> 2;  // the row tile this warp packs
      if (pt < nT) {
        const int i_rel = pt * 128 + quad * 32 + (tid & 31);  // chunk-relative row
        const int ncol = 128 * (pt + 1);
        for (int c0 = 0; c0 < ncol; c0 += 32) {
          uint32_t f0[16], f1[16];
          ptx::tmem_ld16(tmem + lane_base + TC::scf(pt) + c0, f0);
          ptx::tmem_ld16(tmem + lane_base + TC::scf(pt) + c0 + 16, f1);
          ptx::tmem_ld_wait();
          ptx::reg_fence(f0);
          ptx::reg_fence(f1);
          uint32_t pkd[16];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int j0 = c0 + 2 * e, j1 = c0 + 16 + 2 * e;
            pkd[e] = pack_bf2(j0 <= i_rel ? __uint_as_float(f0[2 * e]) : 0.f,
                              j0 + 1 <= i_rel ? __uint_as_float(f0[2 * e + 1]) : 0.f);
            pkd[8 + e] = pack_bf2(j1 <= i_rel ? __uint_as_float(f1[2 * e]) : 0.f,
                                  j1 + 1 <= i_rel ? __uint_as_float(f1[2 * e + 1]) : 0.f);
          }
          ptx::tmem_st16u(tmem + lane_base + TC::pk(pt) + c0 / 2, pkd);
        }
        ptx::tmem_st_wait();
      }
    }
    ptx::tc_fence_before();
    warp_arrive(&pack_done);
    // u, v and the anchors come from the chunk-jump kernel, two launches
    // back: wait until the preceding grids are complete
    ptx::griddep_wait();
    HeadIn in_next = fetch_head(0);

    // In-chunk cumsum of a steep head (one token per thread, threads < T)
    // into Gs / dts of parity q & 1, for the exact per-element epilogue.
    auto steep_cumsum = [&](int q) {
      const int pb = q & 1, h = hbase + q;
      const unsigned short *dtp = reinterpret_cast<const unsigned short *>(a.dt);
      const unsigned short raw =
          tok_ok && SSD_IN_BOUNDS(h < nh && b < a.nb, a.err, 63)
              ? dtp[((int64_t)b * L + tok0 + tid) * nh + h]
              : (unsigned short)0;
      const float d = __uint_as_float((uint32_t)raw << 16);  // bf16 -> fp32, exact
      float incl = a.A[h] * kLog2e * d;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, incl, off);
        if ((tid & 31) >= off) incl += o;
      }
      if ((tid & 31) == 31) warp_tot[warp] = incl;
      ptx::named_bar_sync(1, kRowThreads);
      float Gj = incl;
#pragma unroll
      for (int w2 = 0; w2 < kRowWarps; ++w2)
        if (w2 < warp) Gj += warp_tot[w2];
      if (tid < kT) {
        Gs[pb][tid] = Gj;
        dts[pb][tid] = d;
      }
      ptx::named_bar_sync(1, kRowThreads);
    };

    // The epilogue of head q (inputs `in`, raw x row segment `xk`; u_x =
    // the head's first x stage, read raw only on the steep path):
    // y = u_i Acc_i + D x_i, staged and stored by TMA.
    auto epilogue = [&](int q, int u_x, const HeadIn &in, const uint4 (&xk)[kCols / 8]) {
      const int pb = q & 1, set = q & 1, h = hbase + q;
      ptx::mbar_wait(&acc_full[set], (q >> 1) & 1, a.err, 150);
      ptx::tc_fence_after();
      uint32_t acc[kCols];
#pragma unroll
      for (int c = 0; c < kCols / 16; ++c)
        ptx::tmem_ld16(tmem + lane_base + TC::acc(set, etile) + ecol + 16 * c,
                       *reinterpret_cast<uint32_t(*)[16]>(acc + 16 * c));
      ptx::tmem_ld_wait();
      ptx::reg_fence(acc);
      ptx::tc_fence_before();
      warp_arrive(&acc_free[set]);  // the accumulators may take head q + 2
      float yv[kCols];
      if (!in.steep) {
#pragma unroll
        for (int m = 0; m < kCols / 8; ++m) {
          float xv[8];
          unpack16(xk[m], xv, (__nv_bfloat16 *)nullptr);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            yv[8 * m + e] = fmaf(in.D, xv[e], in.u * __uint_as_float(acc[8 * m + e]));
        }
      } else {
        // exact per-element path: the inter-chunk term from the accumulator
        // (the stored state of a steep chunk is unscaled: plain C h^T), the
        // in-chunk sum on the CUDA cores from the packed masked C B^T (this
        // row's lane) and the raw x rows
        const float Gi = Gs[pb][erow];
        const float ei = exp2f(Gi);
#pragma unroll
        for (int c = 0; c < kCols; ++c) yv[c] = ei * __uint_as_float(acc[c]);
        // packed columns of the row's tile cover tokens 0 .. 128 (etile + 1) - 1
        const int jmax_warp = (kT == 256 ? (warp >> 2) * 128 + (quad * 32) + 31 : quad * 32 + 31);
        for (int j0 = 0; j0 <= jmax_warp; j0 += 32) {
          uint32_t cb[16];
          ptx::tmem_ld16(tmem + lane_base + TC::pk(etile) + j0 / 2, cb);
          ptx::tmem_ld_wait();
          ptx::reg_fence(cb);
          for (int e = 0; e < 32; ++e) {
            const int j = j0 + e;
            if (j > erow) break;
            const uint32_t w = cb[e >> 1];
            const float cbij = __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
            const float s = cbij * exp2f(Gi - Gs[pb][j]) * dts[pb][j];
            const uint8_t *xr = slot_ptr(u_x + (j >> 7));
#pragma unroll
            for (int m = 0; m < kCols / 8; ++m) {
              float xv[8];
              unpack16(*reinterpret_cast<const uint4 *>(
                           xr + sw128(j & 127, ((ecol >> 3) + m) * 16)),
                       xv, (__nv_bfloat16 *)nullptr);
#pragma unroll
              for (int e2 = 0; e2 < 8; ++e2) yv[8 * m + e2] = fmaf(s, xv[e2], yv[8 * m + e2]);
            }
          }
        }
#pragma unroll
        for (int m = 0; m < kCols / 8; ++m) {
          float xv[8];
          unpack16(xk[m], xv, (__nv_bfloat16 *)nullptr);
#pragma unroll
          for (int e = 0; e < 8; ++e) yv[8 * m + e] = fmaf(in.D, xv[e], yv[8 * m + e]);
        }
        // every thread has read the raw x stages: they may be refilled
        ptx::named_bar_sync(2, kRowThreads);
        if (tid == 0)
          for (int xt = 0; xt < nT; ++xt) ptx::mbar_arrive(&empty[(u_x + xt) % nslot]);
      }
      // y through the staging buffer(s), stored by TMA (rows past the
      // sequence are clipped by the store); the previous store must have
      // read the buffer first
      const int nyst = a.nyst;
      for (int t = 0; t < nT; ++t) {
        if (nyst == nT && t > 0) break;  // every tile staged at once
        const bool mine = nyst == nT || etile == t;
        if (tid == 0) ptx::bulk_wait_read<0>();
        ptx::named_bar_sync(2, kRowThreads);
        if (mine) {
          uint8_t *yt = ystage + (nyst == nT ? etile : 0) * kStage;
#pragma unroll
          for (int m = 0; m < kCols / 8; ++m)
            *reinterpret_cast<uint4 *>(yt + sw128(lrow, ((ecol >> 3) + m) * 16)) =
                pack_io16(yv + 8 * m, (__nv_bfloat16 *)nullptr);
        }
        ptx::fence_async_smem();
        ptx::named_bar_sync(2, kRowThreads);
        if (tid == 0) {
          if (nyst == nT) {
            for (int t2 = 0; t2 < nT; ++t2)
              ptx::tma_store_4d(&tm_y, ystage + t2 * kStage, 0, h, tok0 + t2 * 128, b);
          } else {
            ptx::tma_store_4d(&tm_y, ystage, 0, h, tok0 + t * 128, b);
          }
          ptx::bulk_commit();
        }
      }
    };

    // Per head q: scale its x stages (each row times v_j; kept raw for a
    // steep head) keeping this thread's raw segment for D x, then the
    // previous head's epilogue (head q's MMAs overlap it).  A steep head's
    // own epilogue follows at once, so its raw x stages are freed before the
    // ring needs them again.
    int u = n_p1;
    uint32_t xpar = 0;  // parity of the next wait on xfull[slot], one bit per slot
    uint4 xk_prev[kCols / 8];
    HeadIn in_prev{};
    int u_prev = 0;
    bool pending = false;
    for (int q = 0; q < hs; ++q) {
      const HeadIn in = in_next;
      if (q + 1 < hs) in_next = fetch_head(q + 1);
      u += nH;  // the state stages go straight to the MMA warp
      const int u_x = u;
      uint4 xk[kCols / 8];
      for (int xt = 0; xt < nT; ++xt, ++u) {
        const int sl = u % nslot;
        ptx::mbar_wait(&xfull[sl], (xpar >> sl) & 1, a.err, 152);
        xpar ^= 1u << sl;
        if (etile == xt) {
          uint8_t *xs = slot_ptr(u);
#pragma unroll
          for (int m = 0; m < kCols / 8; ++m)
            xk[m] = *reinterpret_cast<const uint4 *>(xs + sw128(lrow, ((ecol >> 3) + m) * 16));
          if (!in.steep) {
#pragma unroll
            for (int m = 0; m < kCols / 8; ++m) {
              float xv[8];
              unpack16(xk[m], xv, (__nv_bfloat16 *)nullptr);
#pragma unroll
              for (int e = 0; e < 8; ++e) xv[e] *= in.v;
              *reinterpret_cast<uint4 *>(xs + sw128(lrow, ((ecol >> 3) + m) * 16)) =
                  pack_io16(xv, (__nv_bfloat16 *)nullptr);
            }
          }
        }
        ptx::fence_async_smem();
        warp_arrive(&scaled[sl]);
      }
      if (pending) epilogue(q - 1, u_prev, in_prev, xk_prev);
      if (in.steep) {
        steep_cumsum(q);
        epilogue(q, u_x, in, xk);
        pending = false;
      } else {
#pragma unroll
        for (int m = 0; m < kCols / 8; ++m) xk_prev[m] = xk[m];
        in_prev = in;
        u_prev = u_x;
        pending = true;
      }
    }
    if (pending) epilogue(hs - 1, u_prev, in_prev, xk_prev);
    if (tid == 0) ptx::bulk_wait<0>();  // every y store complete
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, TC::kAlloc);
}

struct OutSmem {
  int nslot, nyst, smem;
};
// C of the chunk, the ring and the y staging within 220 KB of dynamic shared
// memory (1 KB of it alignment slack; the static arrays, about 6 KB, sit
// beside it): y staging for every row tile when at least a head's stages
// (plus one) still fit the ring, else one staging tile.
OutSmem out_smem(const Dims &d) {
  OutSmem m;
  const int nT = (int)(d.T / 128), nH = (int)((d.S + 127) / 128);
  const int c_bytes = (int)(d.T * d.S * 2);
  const int room = (220 * 1024 - 1024 - c_bytes) / kStage;  // 16 KB units
  m.nyst = room - nT >= nT + nH + 1 ? nT : 1;
  m.nslot = std::min<int>(kMaxSlots, room - m.nyst);
  m.smem = c_bytes + (m.nslot + m.nyst) * kStage + 1024;
  return m;
}

}  // namespace

bool fwd_out_supported(const Dims &d) {
  if (d.P != kP || d.S % 64 || d.S > 256 || (d.T != 128 && d.T != 256)) return false;
  if (d.nc > 65535 || d.b > 65535) return false;
  // the ring must hold a steep head's x stages (released only by its
  // epilogue) and the next head's state stages, or the row warps' order
  // could stall it
  const int need = (int)(d.T / 128 + (d.S + 127) / 128);
  return out_smem(d).nslot >= need;
}

bool fwd_out_heads_ok(const Dims &d, int hs) {
  return fwd_out_supported(d) && hs >= 1 && hs <= d.hpg && d.hpg % hs == 0 &&
         d.nh / hs <= 65535;
}

// Heads per CTA: the divisor of the heads per group minimising the bytes
// the busiest SM moves (waves of CTAs times a CTA's loads and stores: C and
// B of the chunk once, and per head its state, x and y).
int fwd_out_heads(const Dims &d) {
  const int64_t sms = sm_count();
  int best = 1;
  double best_cost = 1e300;
  for (int hs = 1; hs <= d.hpg; ++hs) {
    if (!fwd_out_heads_ok(d, hs)) continue;
    const int64_t ctas = d.b * d.nc * (d.nh / hs);
    const double per_cta = 2.0 * d.T * d.S * 2 + hs * (d.S * 64.0 * 2 + 2.0 * d.T * 64 * 2);
    const double cost = (double)((ctas + sms - 1) / sms) * per_cta;
    if (cost < best_cost * 0.999) {
      best_cost = cost;
      best = hs;
    }
  }
  return best;
}

cudaError_t launch_fwd_out(const Dims &d, const void *x, const void *B, const void *C,
                           const void *dt, const float *A, const void *states, const float *D,
                           const float *u, const float *v, const float2 *anchor, void *y,
                           int hs, int *err, cudaStream_t st) {
  if (!fwd_out_heads_ok(d, hs)) return cudaErrorInvalidValue;
  CUtensorMap tC, tB, tx, tS, tY;
  if (!make_tmap_bl(&tC, C, true, d.b, d.L, d.ng, d.S, 128) ||
      !make_tmap_bl(&tB, B, true, d.b, d.L, d.ng, d.S, 128) ||
      !make_tmap_bl(&tx, x, true, d.b, d.L, d.nh, d.P, 128) ||
      !make_tmap_bl(&tY, y, true, d.b, d.L, d.nh, d.P, 128))
    return cudaErrorInvalidValue;
  {
    // start states as [b * nh * nc][S][P] bf16; one box = up to 128 rows of S
    const uint64_t dims[3] = {(uint64_t)d.P, (uint64_t)d.S, (uint64_t)(d.b * d.nh * d.nc)};
    const uint64_t strides[2] = {(uint64_t)d.P * 2, (uint64_t)(d.S * d.P * 2)};
    const uint32_t box[3] = {64u, (uint32_t)std::min<int64_t>(d.S, 128), 1u};
    if (!make_tmap_sw128(&tS, states, true, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  const OutSmem m = out_smem(d);
  auto kernel = d.T == 256 ? fwd_out_bf16<256> : fwd_out_bf16<128>;
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, m.smem);
  if (e != cudaSuccess) return e;
  OutArgs a;
  a.dt = static_cast<const __nv_bfloat16 *>(dt);
  a.A = A;
  a.D = D;
  a.u = u;
  a.v = v;
  a.anchor = anchor;
  a.err = err;
  a.L = (int)d.L;
  a.nh = (int)d.nh;
  a.S = (int)d.S;
  a.hpg = (int)d.hpg;
  a.T = (int)d.T;
  a.nc = (int)d.nc;
  a.nb = (int)d.b;
  a.hs = hs;
  a.nslot = m.nslot;
  a.nyst = m.nyst;
  // programmatic stream serialisation: the producer waits on the device
  // before loading the first start state
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(d.nh / hs), (unsigned)d.nc, (unsigned)d.b);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = m.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, tC, tB, tx, tS, tY, a);
}

}  // namespace ssd
