// Forward path, output pass (bf16 I/O) with the interaction tile of a chunk
// computed once and shared by a slice of heads.  Same equation as
// fwd_scan.cu (the page's compute_out, chunked output equation of
// "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA
// CUDA Tile", section "Mamba-2 architecture"):
//
//   y_i = exp2(G_i) (h_k c_i) + sum_{j<=i in chunk} (c_i . B_j) exp2(G_i - G_j) dt_j x_j
//         + D x_i
//
// The heads of one group share B and C, so C B^T of a chunk is the same for
// all of them.  One CTA per (slice of hs heads of one group, chunk, batch)
// or, with kSplit, per (slice, 128-row tile of a chunk, batch):
//   phase 1: Sc = C B^T of the CTA's row tiles into tensor memory in fp32,
//            from C resident in shared memory and B resident too (whole
//            chunk) or streamed through a two-slot ring in the second head
//            buffer (kSplit, which is what lets S = 256 fit), then re-packed
//            by the row warps as fp16 pairs (half the columns);
//   per head q of the slice (state and x tiles double-buffered, so the next
//            head's loads overlap this head):
//            Yc = C h_q^T for each row tile, the decayed, masked tile S'_q
//            from Sc written to tensor memory as bf16 pairs one 64-token
//            block at a time (two stages), Ys = S'_q X_q with S'_q read from
//            tensor memory, and the epilogue, row tile by row tile,
//            y = exp2(G_i) Yc + Ys + D x computed over x in shared memory and
//            written by TMA stores (the next head's cumsum runs while this
//            head's last MMAs finish).  y may overwrite x only once every
//            S'_q X_q product of the head has completed.
// Warp roles: warp 8 loads (TMA), warp 9 issues the MMAs, warps 0-7 do the
// cumsums, the re-packing, the decay and the epilogue (two warps per 32-lane
// quadrant, each taking 32 of every 64 columns).
//
// Supported: P = 64; S in {64, 128} with T in {128, 256}, and with kSplit S
// up to 256; other shapes use fwd_scan.cu.  The decay factors are those of
// fwd_scan.cu: for a 64-token column block ending at r strictly before row
// i's block, exp2(G_i - G_j) = exp2(G_i - G_r) * exp2(G_r - G_j), both
// exponents <= 0; the row's own block uses the same factors when its total
// decay is bounded (see kSpanMax).
#include <cuda_fp16.h>

#include "fwd.cuh"

namespace ssd {
namespace {

constexpr int kRowWarps = 8;
constexpr int kRowThreads = kRowWarps * 32;
// column split of every 64-column block between the row warps of a TMEM
// lane quadrant: kCG groups of kCPT columns (kC16 16-column loads, kCH
// 16-byte chunks of a 128-byte smem row)
constexpr int kCG = kRowWarps / 4;
constexpr int kCPT = 64 / kCG;
constexpr int kC16 = kCPT / 16;
constexpr int kCH = kCPT / 8;
constexpr int kThreads = kRowThreads + 64;
constexpr int kProducerWarp = kRowWarps, kMmaWarp = kRowWarps + 1;
constexpr int kP = 64;              // head dimension handled here
constexpr int kNP = 2;              // stages of the decayed interaction tile S'
constexpr int kBlk = 64 * 128;      // 64 rows of 128 bytes
constexpr int kTile = 128 * 128;    // 128 rows of 128 bytes
// packed (two-column) tensor-memory columns of a thread's part of a block
constexpr int kPP = kCPT / 2;
static_assert(kCPT == 32 || kCPT == 16, "a thread's S' row segment is one 8- or 16-column store");
// Tensor-memory columns.  Phase 1 accumulates C B^T in fp32 (row tile 1:
// [0, 256), row tile 0: [256, 384)); the row warps re-pack it as fp16 pairs
// (row tile 1: [256, 384), row tile 0: [384, 448)), which frees the rest for
// the two accumulators of a head, Ys = S' X (row tile t at 64 t) and
// Yc = C h^T (row tile 0 at 192, row tile 1 at 448), and the two stages of
// the decayed tile S' as bf16 pairs, the A operand of the S' X MMAs ([128,
// 160), [160, 192)).  The epilogue combines y = exp2(G_i) Yc + Ys + D x.
__device__ __forceinline__ uint32_t ys_col(int t) { return 64u * (uint32_t)t; }
__device__ __forceinline__ uint32_t yc_col(int t) { return t ? 448u : 192u; }
__device__ __forceinline__ uint32_t scf_col(int t) { return t ? 0u : 256u; }
__device__ __forceinline__ uint32_t sch_col(int t) { return t ? 256u : 384u; }
__device__ __forceinline__ uint32_t sp_col(int s) { return 128u + 32u * (uint32_t)s; }

// The fp16 copy of C B^T holds 2^-4 C B^T: magnitudes up to 2^20 stay
// finite, and values below 2^-10 (subnormal) keep an absolute error of at
// most 2^-21.  The decay factors carry the 2^4 back.
constexpr float kScDown = 0.0625f, kScUp = 16.f, kScUpLog2 = 4.f;
// Largest total decay (log2 units, the sum of -A dt log2(e) over a 64-token
// block) for which the row's own block uses the factored decay.
constexpr float kSpanMax = 96.f;
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo * kScDown, hi * kScDown);
  return *reinterpret_cast<const uint32_t *>(&h);
}
__device__ __forceinline__ float2 unpack_h2(uint32_t u) {
  return __half22float2(*reinterpret_cast<const __half2 *>(&u));
}
__device__ __forceinline__ uint32_t pack_bf2(float2 v) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(v.x, v.y);
  return *reinterpret_cast<const uint32_t *>(&b);
}

struct ChunkArgs {
  const __nv_bfloat16 *x, *dt;
  const float *A, *D;
  __nv_bfloat16 *y;
  int *err;
  int L, nh, S, hpg, T, nc, hs;
  int nb;  // batch count (the extents the debug-bounds checks use)
  // shared-memory layout (byte offsets from the 1024-aligned base)
  int off_C, off_B, off_hx0, off_hx1;
};

template <bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
fwd_scan_chunk_bf16(const __grid_constant__ CUtensorMap tm_C,
                    const __grid_constant__ CUtensorMap tm_B,
                    const __grid_constant__ CUtensorMap tm_x,
                    const __grid_constant__ CUtensorMap tm_st,
                    const __grid_constant__ CUtensorMap tm_y, const ChunkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t p1_full[2], p1_empty[2], sc_done, pack_done, hx_full[2],
      hx_empty[2],
      pm_full[kNP], pm_empty[kNP], ydone, yfree[2];
  __shared__ uint32_t tmem_slot;
  // per head (double-buffered by head parity): G in log2 units, dt, and the
  // column factors v_j = exp2(G_r - G_j) dt_j of the factored decay; read
  // with 16-byte vector loads, so each array is 16-byte aligned
  __shared__ __align__(16) float Gs[2][256];
  __shared__ __align__(16) float dts[2][256];
  __shared__ __align__(16) float vs[2][256];
  __shared__ float warp_tot[2][8];

  const int L = a.L, nh = a.nh, S = a.S, T = a.T, nc = a.nc, hs = a.hs;
  const int tid = threadIdx.x, warp = tid >> 5;
  constexpr bool split = kSplit;
  const int ntile_all = T / 128;
  const int k = split ? blockIdx.y / ntile_all : blockIdx.y, b = blockIdx.z;
  // the row tiles [t_lo, t_hi) of the chunk this CTA computes
  const int t_lo = split ? blockIdx.y % ntile_all : 0;
  const int t_hi = split ? t_lo + 1 : ntile_all;
  const int hbase = blockIdx.x * hs, g = hbase / a.hpg;
  const int tok0 = k * T;
  const int valid = min(T, L - tok0);
  const int nsb = S / 64;
  const int st_bytes = S * kP * 2;
  // a head's tiles: its start state, then x rows 0 .. 128 t_hi - 1
  const int hx_bytes = st_bytes + t_hi * 2 * kBlk;
  // C rows of this CTA's tiles, per 64-wide block of S
  auto c_off = [&](int t, int sb) { return a.off_C + ((t - t_lo) * nsb + sb) * kTile; };
  const uint32_t ncols = 512;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&p1_full[i], 1);
      ptx::mbar_init(&p1_empty[i], 1);
      ptx::mbar_init(&hx_full[i], 1);
      ptx::mbar_init(&hx_empty[i], 2);  // MMA commit + the y store has read the tile
    }
    ptx::mbar_init(&sc_done, 1);
    // the row warps arrive once per warp (lane 0, after __syncwarp)
    ptx::mbar_init(&pack_done, kRowWarps);
    for (int i = 0; i < kNP; ++i) {
      ptx::mbar_init(&pm_full[i], kRowWarps);
      ptx::mbar_init(&pm_empty[i], 1);
    }
    ptx::mbar_init(&ydone, 1);
    ptx::mbar_init(&yfree[0], kRowWarps);  // per row tile
    ptx::mbar_init(&yfree[1], kRowWarps);
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(&tmem_slot, ncols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const bool leader = (tid & 31) == 0;
  // second head buffer reuses B's space (resident B) or holds the B ring
  const bool alias_hx1 = split || a.off_hx1 == a.off_B;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // phase 1, one 64-wide block sb of S at a time: C rows of this CTA's
    // tiles and B rows 0 .. 128 t_hi - 1.  Resident B: every block at once.
    // Split: B block sb into ring slot sb & 1 (in the second head buffer),
    // once the MMAs of block sb - 2 are done; blocks 2 and up are issued
    // after head 0's loads, which need no slot
    auto load_p1 = [&](int sb) {
      const int slot = split ? (sb & 1) : sb;
      if (split && sb >= 2) ptx::mbar_wait(&p1_empty[slot], ((sb >> 1) - 1) & 1, a.err, 120);
      if (leader) {
        ptx::mbar_arrive_expect_tx(&p1_full[slot], (t_hi - t_lo + t_hi) * kTile);
        for (int t = t_lo; t < t_hi; ++t)
          ptx::tma_load_4d(smem + c_off(t, sb), &tm_C, sb * 64, g, tok0 + t * 128, b,
                           &p1_full[slot]);
        uint8_t *bdst = split ? smem + a.off_hx1 + slot * 2 * kTile
                              : smem + a.off_B + sb * ntile_all * kTile;
        for (int t = 0; t < t_hi; ++t)
          ptx::tma_load_4d(bdst + t * kTile, &tm_B, sb * 64, g, tok0 + t * 128, b,
                           &p1_full[slot]);
      }
      __syncwarp();
    };
    const int nsb_first = split ? min(nsb, 2) : nsb;
    for (int sb = 0; sb < nsb_first; ++sb) load_p1(sb);
    for (int q = 0; q < hs; ++q) {
      const int buf = q & 1;
      if (q == 1)
        for (int sb = nsb_first; sb < nsb; ++sb) load_p1(sb);
      ptx::mbar_wait(&hx_empty[buf], ((q >> 1) & 1) ^ 1, a.err, 121);
      if (q == 1 && alias_hx1) ptx::mbar_wait(&sc_done, 0, a.err, 122);
      if (leader) {
        uint8_t *hx = smem + (buf ? a.off_hx1 : a.off_hx0);
        ptx::mbar_arrive_expect_tx(&hx_full[buf], hx_bytes);
        // x rows of the chunk (64-token blocks, p contiguous)
        for (int jb = 0; jb < 2 * t_hi; ++jb)
          ptx::tma_load_4d(hx + st_bytes + jb * kBlk, &tm_x, 0, hbase + q, tok0 + jb * 64, b,
                           &hx_full[buf]);
        // the start state comes from the preceding kernel (the state pass),
        // which may still be running when this CTA starts
        if (q == 0) ptx::griddep_wait();
        const int row = (b * nh + hbase + q) * nc + k;
        for (int sb = 0; sb < nsb; ++sb)
          ptx::tma_load_3d(hx + sb * kBlk, &tm_st, 0, sb * 64, row, &hx_full[buf]);
      }
      __syncwarp();
    }
    if (hs == 1)
      for (int sb = nsb_first; sb < nsb; ++sb) load_p1(sb);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // phase 1: Sc = C B^T; row tile t needs columns j < 128 (t + 1)
    for (int sb = 0; sb < nsb; ++sb) {
      const int slot = split ? (sb & 1) : sb;
      ptx::mbar_wait(&p1_full[slot], split ? (sb >> 1) & 1 : 0, a.err, 123);
      ptx::tc_fence_after();
      if (leader) {
        const uint32_t b0 = ptx::smem_u32(split ? smem + a.off_hx1 + slot * 2 * kTile
                                                : smem + a.off_B + sb * ntile_all * kTile);
        for (int t = t_lo; t < t_hi; ++t) {
          const uint32_t c0 = ptx::smem_u32(smem + c_off(t, sb));
          const uint32_t idS = ptx::idesc_bf16(128, 128 * (t + 1), false, false);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t cd = ptx::smem_desc(c0 + kk * 32, 16, 1024, ptx::kSw128);
            const uint64_t bd = ptx::smem_desc(b0 + kk * 32, 16, 1024, ptx::kSw128);
            ptx::mma_ss<false>(tmem + scf_col(t), cd, bd, idS, (sb | kk) ? 1u : 0u);
          }
        }
        if (split) ptx::mma_commit(&p1_empty[slot]);
      }
      __syncwarp();
    }
    if (leader) ptx::mma_commit(&sc_done);
    __syncwarp();
    const uint32_t idY = ptx::idesc_bf16(128, kP, false, true);
    // the accumulators and the S' stages overlap the fp32 C B^T: wait for
    // its re-packing
    ptx::mbar_wait(&pack_done, 0, a.err, 133);
    int cnt = 0;  // S' blocks consumed so far
    for (int q = 0; q < hs; ++q) {
      const int buf = q & 1;
      const uint32_t hx = ptx::smem_u32(smem + (buf ? a.off_hx1 : a.off_hx0));
      ptx::mbar_wait(&hx_full[buf], (q >> 1) & 1, a.err, 124);
      // Yc = C h_q^T for each row tile, once the previous head's epilogue
      // has read that tile's accumulators
      for (int t = t_lo; t < t_hi; ++t) {
        if (q > 0) ptx::mbar_wait(&yfree[t], (q - 1) & 1, a.err, 125);
        ptx::tc_fence_after();
        if (leader) {
          for (int sb = 0; sb < nsb; ++sb) {
            const uint32_t c0 = ptx::smem_u32(smem + c_off(t, sb));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t cd = ptx::smem_desc(c0 + kk * 32, 16, 1024, ptx::kSw128);
              const uint64_t hd =
                  ptx::smem_desc(hx + sb * kBlk + kk * 2048, kBlk, 1024, ptx::kSw128);
              ptx::mma_ss<false>(tmem + yc_col(t), cd, hd, idY, (sb | kk) ? 1u : 0u);
            }
          }
        }
        __syncwarp();
      }
      // Ys = S'_q X_q, one 64-token block of each row tile at a time
      for (int t = t_lo; t < t_hi; ++t)
        for (int jb = 0; jb < 2 * (t + 1); ++jb, ++cnt) {
          const int s = cnt % kNP;
          ptx::mbar_wait(&pm_full[s], (cnt / kNP) & 1, a.err, 127);
          ptx::tc_fence_after();
          if (leader) {
            const uint32_t x0 = hx + st_bytes + jb * kBlk;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t xd = ptx::smem_desc(x0 + kk * 2048, kBlk, 1024, ptx::kSw128);
              ptx::mma_ts_bf16(tmem + ys_col(t), tmem + sp_col(s) + kk * 8, xd, idY,
                               (jb | kk) ? 1u : 0u);
            }
            ptx::mma_commit(&pm_empty[s]);
          }
          __syncwarp();
        }
      if (leader) {
        ptx::mma_commit(&ydone);
        ptx::mma_commit(&hx_empty[buf]);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ row warps
    const int quad = warp & 3, cg = warp >> 2;  // TMEM lane quadrant, column group
    const int r = quad * 32 + (tid & 31);       // row within a tile = TMEM lane
    const int c32 = cg * kCPT;                  // this thread's columns of a 64-block
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;

    // dt of the next head for token tid (tid < T), as raw bf16 bits until
    // the cumsum uses it, so no instruction waits on the load before then
    const unsigned short *dtp = reinterpret_cast<const unsigned short *>(a.dt);
    const bool tok_ok = tid < valid;
    const int64_t dt_off = ((int64_t)b * L + tok0 + (tok_ok ? tid : 0)) * nh + hbase;
    // every head of the slice lies in [0, nh) and b in [0, nb)
    const bool hok = SSD_IN_BOUNDS(hbase + hs <= nh && b < a.nb, a.err, 140);
    unsigned short draw = tok_ok && hok ? dtp[dt_off] : (unsigned short)0;
    float Aq = hok ? a.A[hbase] : 0.f;
    // in-chunk cumsum of head q (one token per thread, threads < T) into the
    // buffers of parity q & 1, and the column factors of the factored decay;
    // then the dt of head q + 1 is fetched
    auto cumsum = [&](int q) {
      const int pb = q & 1;
      const float d = __uint_as_float((uint32_t)draw << 16);  // bf16 -> fp32, exact
      float incl = Aq * kLog2e * d;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, incl, off);
        if ((tid & 31) >= off) incl += o;
      }
      if ((tid & 31) == 31 && warp < 8) warp_tot[pb][warp] = incl;
      ptx::named_bar_sync(1, kRowThreads);
      // G at this token, and at the last token of its 64-token block (the
      // end of warp (warp | 1)), both from the warp totals
      float Gj = incl, Gr = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < 8; ++w2) {
        const float tw = warp_tot[pb][w2];
        if (w2 < warp) Gj += tw;
        if (w2 <= (warp | 1)) Gr += tw;
      }
      if (tid < T) {
        Gs[pb][tid] = Gj;
        dts[pb][tid] = d;
        vs[pb][tid] = ptx::ex2_approx(Gr - Gj) * d;
      }
      ptx::named_bar_sync(1, kRowThreads);
      if (q + 1 < hs) {
        draw = tok_ok && hok ? dtp[dt_off + q + 1] : (unsigned short)0;
        Aq = hok ? a.A[hbase + q + 1] : 0.f;
      }
    };

    ptx::mbar_wait(&sc_done, 0, a.err, 128);
    ptx::tc_fence_after();
    // re-pack the fp32 C B^T as fp16 pairs (at most 2^-11 relative rounding
    // before the decay, well below the bf16 rounding of S'), row tile 0
    // first: its fp32 columns are then overwritten by row tile 1's copy
    for (int t = t_lo; t < t_hi; ++t) {
      if (t > t_lo) {
        ptx::tc_fence_before();
        ptx::named_bar_sync(1, kRowThreads);  // every thread has read tile 0's fp32
        ptx::tc_fence_after();
      }
      for (int jb = 0; jb < 2 * (t + 1); ++jb) {
        uint32_t f[kC16][16];
#pragma unroll
        for (int c = 0; c < kC16; ++c)
          ptx::tmem_ld16(tmem + lane_base + scf_col(t) + jb * 64 + c32 + c * 16, f[c]);
        ptx::tmem_ld_wait();
        uint32_t hv[kPP];
#pragma unroll
        for (int c = 0; c < kC16; ++c) {
          ptx::reg_fence(f[c]);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            hv[c * 8 + e] = pack_h2(__uint_as_float(f[c][2 * e]), __uint_as_float(f[c][2 * e + 1]));
        }
        ptx::tmem_stu<kPP>(tmem + lane_base + sch_col(t) + jb * 32 + cg * kPP, hv);
      }
    }
    ptx::tmem_st_wait();
    ptx::tc_fence_before();
    __syncwarp();
    if ((tid & 31) == 0) ptx::mbar_arrive(&pack_done);
    cumsum(0);
    int cnt = 0;
    for (int q = 0; q < hs; ++q) {
      const int pb = q & 1, buf = q & 1;
      const int h = hbase + q;
      const float Dh = a.D ? a.D[h] : 0.f;  // used in the epilogue: load it early


      // decayed, masked interaction rows, one 64-token block (one S' stage)
      // per tensor-memory load wait
      for (int t = t_lo; t < t_hi; ++t) {
        const int i_rel = t * 128 + r;
        const int rb = i_rel >> 6;
        const float Git = Gs[pb][i_rel];
        const float Git4 = Git + kScUpLog2;  // exp2(Git4 - G_j) = 2^4 exp2(Git - G_j)
        for (int jb = 0; jb < 2 * (t + 1); ++jb, ++cnt) {
          // pu: this thread's kCPT columns of S' as kPP bf16 pairs, the even
          // column in the low half (blocks right of the row's block are 0)
          uint32_t pu[kPP];
          if (jb <= rb) {
            // the same columns of C B^T, as fp16 pairs
            uint32_t sh[kPP];
            ptx::tmem_ldu<kPP>(tmem + lane_base + sch_col(t) + jb * 32 + cg * kPP, sh);
            ptx::tmem_ld_wait();
            ptx::reg_fence(sh);
            if (jb < rb) {
              // whole block before the row's block: factored decay
              const float ui = kScUp * ptx::ex2_approx(Git - Gs[pb][jb * 64 + 63]);
              const float2 ui2 = make_float2(ui, ui);
              const float4 *vp = reinterpret_cast<const float4 *>(&vs[pb][jb * 64 + c32]);
#pragma unroll
              for (int m = 0; m < kCPT / 4; ++m) {
                const float4 f = vp[m];
                const float2 w0 = ptx::mul_f32x2(make_float2(f.x, f.y), ui2);
                const float2 w1 = ptx::mul_f32x2(make_float2(f.z, f.w), ui2);
                pu[2 * m] = pack_bf2(ptx::mul_f32x2(unpack_h2(sh[2 * m]), w0));
                pu[2 * m + 1] = pack_bf2(ptx::mul_f32x2(unpack_h2(sh[2 * m + 1]), w1));
              }
            } else if (-(warp_tot[pb][2 * jb] + warp_tot[pb][2 * jb + 1]) < kSpanMax) {
              // the row's own block, whose total decay exp2(-span) is above
              // 2^-kSpanMax: the same factors about its last token r, now
              // exp2(G_i - G_r) <= 2^kSpanMax and exp2(G_r - G_j) >= 2^-kSpanMax
              // (no overflow, no underflow), with the causal mask: columns
              // k <= klim of the thread's kCPT are kept (j <= i, j < valid)
              const int klim = min(i_rel, valid - 1) - (jb * 64 + c32);
              const float ui = kScUp * ptx::ex2_approx(Git - Gs[pb][jb * 64 + 63]);
              const float2 ui2 = make_float2(ui, ui);
              const float4 *vp = reinterpret_cast<const float4 *>(&vs[pb][jb * 64 + c32]);
#pragma unroll
              for (int m = 0; m < kCPT / 4; ++m) {
                const float4 f = vp[m];
                const float2 w0 = ptx::mul_f32x2(make_float2(f.x, f.y), ui2);
                const float2 w1 = ptx::mul_f32x2(make_float2(f.z, f.w), ui2);
                float2 v0 = ptx::mul_f32x2(unpack_h2(sh[2 * m]), w0);
                float2 v1 = ptx::mul_f32x2(unpack_h2(sh[2 * m + 1]), w1);
                v0.x = 4 * m + 0 <= klim ? v0.x : 0.f;
                v0.y = 4 * m + 1 <= klim ? v0.y : 0.f;
                v1.x = 4 * m + 2 <= klim ? v1.x : 0.f;
                v1.y = 4 * m + 3 <= klim ? v1.y : 0.f;
                pu[2 * m] = pack_bf2(v0);
                pu[2 * m + 1] = pack_bf2(v1);
              }
            } else {
              // the row's own block with a steep decay: direct exponent,
              // causal mask (columns k <= klim kept, as above)
              const int klim = min(i_rel, valid - 1) - (jb * 64 + c32);
              const float4 *gp = reinterpret_cast<const float4 *>(&Gs[pb][jb * 64 + c32]);
              const float4 *dp = reinterpret_cast<const float4 *>(&dts[pb][jb * 64 + c32]);
              const float2 g2 = make_float2(Git4, Git4);
#pragma unroll
              for (int m = 0; m < kCPT / 4; ++m) {
                const float4 gj = gp[m], dj = dp[m];
                float2 e0 = ptx::sub_f32x2(g2, make_float2(gj.x, gj.y));
                float2 e1 = ptx::sub_f32x2(g2, make_float2(gj.z, gj.w));
                e0 = make_float2(ptx::ex2_approx(e0.x), ptx::ex2_approx(e0.y));
                e1 = make_float2(ptx::ex2_approx(e1.x), ptx::ex2_approx(e1.y));
                float2 v0 = ptx::mul_f32x2(ptx::mul_f32x2(unpack_h2(sh[2 * m]), e0),
                                           make_float2(dj.x, dj.y));
                float2 v1 = ptx::mul_f32x2(ptx::mul_f32x2(unpack_h2(sh[2 * m + 1]), e1),
                                           make_float2(dj.z, dj.w));
                v0.x = 4 * m + 0 <= klim ? v0.x : 0.f;
                v0.y = 4 * m + 1 <= klim ? v0.y : 0.f;
                v1.x = 4 * m + 2 <= klim ? v1.x : 0.f;
                v1.y = 4 * m + 3 <= klim ? v1.y : 0.f;
                pu[2 * m] = pack_bf2(v0);
                pu[2 * m + 1] = pack_bf2(v1);
              }
            }
          } else {
#pragma unroll
            for (int m = 0; m < kPP; ++m) pu[m] = 0u;
          }
          // into tensor-memory stage s as 16 columns of bf16 pairs (the even
          // column in the low half), the A operand of the S' X MMA
          const int s = cnt % kNP;
          ptx::mbar_wait(&pm_empty[s], ((cnt / kNP) & 1) ^ 1, a.err, 130);
          ptx::tc_fence_after();
          ptx::tmem_stu<kPP>(tmem + lane_base + sp_col(s) + cg * kPP, pu);
          ptx::tmem_st_wait();
          ptx::tc_fence_before();
          __syncwarp();
          if ((tid & 31) == 0) ptx::mbar_arrive(&pm_full[s]);
          // the previous head's y store has had the first row tile's time to
          // read its shared-memory tile: release that head buffer
          if (tid == 0 && q > 0 && t == t_lo && jb == 1) {
            ptx::bulk_wait_read<0>();
            ptx::mbar_arrive(&hx_empty[(q - 1) & 1]);
          }
        }
      }

      // the next head's cumsum while this head's last MMAs finish
      if (q + 1 < hs) cumsum(q + 1);

      // epilogue: y = exp2(G_i) Yc + Ys + D x, written over x in the head's
      // shared-memory tile and stored by TMA
      ptx::mbar_wait(&ydone, q & 1, a.err, 131);
      ptx::tc_fence_after();
      uint8_t *xs = smem + (buf ? a.off_hx1 : a.off_hx0) + st_bytes;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (t < t_lo) continue;
        if (t >= t_hi) break;
        const int i_rel = t * 128 + r;
        uint8_t *xrow = xs + (i_rel >> 6) * kBlk;
        uint32_t ys[kC16][16], yc[kC16][16];
#pragma unroll
        for (int c = 0; c < kC16; ++c) {
          ptx::tmem_ld16(tmem + lane_base + ys_col(t) + c32 + c * 16, ys[c]);
          ptx::tmem_ld16(tmem + lane_base + yc_col(t) + c32 + c * 16, yc[c]);
        }
        ptx::tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < kC16; ++c) {
          ptx::reg_fence(ys[c]);
          ptx::reg_fence(yc[c]);
        }
        ptx::tc_fence_before();
        __syncwarp();
        // this row tile's Yc and Ys may now take the next head
        if ((tid & 31) == 0) ptx::mbar_arrive(&yfree[t]);
        const float eg = ptx::ex2_approx(Gs[pb][i_rel]);  // carried-state decay
#pragma unroll
        for (int k4 = 0; k4 < kCH; ++k4) {
          uint4 *p4 = reinterpret_cast<uint4 *>(xrow + sw128(i_rel & 63, (cg * kCH + k4) * 16));
          float xv[8];
          unpack16(*p4, xv, (__nv_bfloat16 *)nullptr);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int c = k4 >> 1, ce = (k4 & 1) * 8 + e;
            xv[e] = fmaf(Dh, xv[e], fmaf(eg, __uint_as_float(yc[c][ce]), __uint_as_float(ys[c][ce])));
          }
          *p4 = pack_io16(xv, (__nv_bfloat16 *)nullptr);
        }
      }
      ptx::fence_async_smem();
      ptx::named_bar_sync(2, kRowThreads);
      if (tid == 0) {
        for (int jb = 2 * t_lo; jb < 2 * t_hi; ++jb)
          ptx::tma_store_4d(&tm_y, xs + jb * kBlk, 0, h, tok0 + jb * 64, b);
        ptx::bulk_commit();
      }
    }
    if (tid == 0) ptx::bulk_wait<0>();  // every y store complete
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, ncols);
}

struct Layout {
  int off_C, off_B, off_hx[2], hx_bytes, total;
};

// Split launches: C of one row tile, then two head buffers of at least
// four 16 KB tiles each (the second one holds the two-slot B ring of
// phase 1).
Layout split_layout(const Dims &d) {
  Layout l;
  const int nsb = (int)(d.S / 64);
  l.hx_bytes = (int)(d.S * kP * 2 + d.T * kP * 2);
  const int buf = std::max(l.hx_bytes, 4 * kTile);
  l.off_C = 0;
  l.off_B = -1;
  l.off_hx[0] = nsb * kTile;
  l.off_hx[1] = l.off_hx[0] + buf;
  l.total = l.off_hx[1] + buf;
  return l;
}

Layout chunk_layout(const Dims &d) {
  Layout l;
  const int ntile = (int)(d.T / 128), nsb = (int)(d.S / 64);
  const int cb = ntile * nsb * kTile;  // C, and B, of the chunk
  l.hx_bytes = (int)(d.S * kP * 2 + d.T * kP * 2);
  l.off_C = 0;
  l.off_B = cb;
  l.off_hx[0] = 2 * cb;
  const int base = l.off_hx[0] + l.hx_bytes;
  if (base + l.hx_bytes <= 200 * 1024) {
    l.off_hx[1] = base;
    l.total = base + l.hx_bytes;
  } else {
    l.off_hx[1] = l.off_B;  // the second head buffer reuses B once phase 1 is done
    l.total = base;
  }
  return l;
}

}  // namespace

bool fwd_scan_chunk_supported(const Dims &d) {
  if (d.P != kP || (d.S != 64 && d.S != 128) || (d.T != 128 && d.T != 256)) return false;
  const Layout l = chunk_layout(d);
  if (l.off_hx[1] == l.off_B && l.hx_bytes > l.off_hx[0] - l.off_B) return false;
  return l.total + 1024 <= 210 * 1024;
}

bool fwd_scan_chunk_split_supported(const Dims &d) {
  if (d.P != kP || (d.S != 64 && d.S != 128 && d.S != 256) || (d.T != 128 && d.T != 256))
    return false;
  if (d.nc * (d.T / 128) > 65535) return false;
  return split_layout(d).total + 1024 <= 210 * 1024;
}

// Heads per CTA: a divisor of the heads per group minimising
// waves * (phase-1 cost + heads), the phase-1 cost counted as one head.
int fwd_scan_chunk_heads(const Dims &d, bool split) {
  const int64_t sms = sm_count();
  int best = 1;
  double best_cost = 1e300;
  for (int hs = 1; hs <= d.hpg; ++hs) {
    if (d.hpg % hs) continue;
    const int64_t ctas = d.b * d.nc * (split ? d.T / 128 : 1) * (d.nh / hs);
    const double cost = (double)((ctas + sms - 1) / sms) * (1.0 + hs);
    if (cost < best_cost * 0.999) {
      best_cost = cost;
      best = hs;
    }
  }
  return best;
}

bool fwd_scan_chunk_heads_ok(const Dims &d, int hs, bool split) {
  return (split ? fwd_scan_chunk_split_supported(d) : fwd_scan_chunk_supported(d)) &&
         hs >= 1 && hs <= d.hpg && d.hpg % hs == 0;
}

cudaError_t launch_fwd_scan_chunk(const Dims &d, const void *x, const void *B, const void *C,
                                  const void *dt, const float *A, const void *states,
                                  const float *D, void *y, int hs, bool split, int *err,
                                  cudaStream_t st) {
  if (!fwd_scan_chunk_heads_ok(d, hs, split)) return cudaErrorInvalidValue;
  CUtensorMap tC, tB, tx, tS, tY;
  if (!make_tmap_bl(&tC, C, true, d.b, d.L, d.ng, d.S, 128) ||
      !make_tmap_bl(&tB, B, true, d.b, d.L, d.ng, d.S, 128) ||
      !make_tmap_bl(&tx, x, true, d.b, d.L, d.nh, d.P, 64) ||
      !make_tmap_bl(&tY, y, true, d.b, d.L, d.nh, d.P, 64))
    return cudaErrorInvalidValue;
  {
    const uint64_t dims[3] = {(uint64_t)d.P, (uint64_t)d.S, (uint64_t)(d.b * d.nh * d.nc)};
    const uint64_t strides[2] = {(uint64_t)d.P * 2, (uint64_t)(d.S * d.P * 2)};
    const uint32_t box[3] = {64u, 64u, 1u};
    if (!make_tmap_sw128(&tS, states, true, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  const Layout l = split ? split_layout(d) : chunk_layout(d);
  const int smem = l.total + 1024;
  // kSplit: one 128-row tile of the chunk per CTA (blockIdx.y = chunk *
  // tiles + tile), B streamed through a two-slot ring in the second head
  // buffer during phase 1; else both row tiles per CTA, B resident
  auto kernel = split ? fwd_scan_chunk_bf16<true> : fwd_scan_chunk_bf16<false>;
  cudaError_t e = cudaFuncSetAttribute(kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  ChunkArgs a;
  a.x = static_cast<const __nv_bfloat16 *>(x);
  a.dt = static_cast<const __nv_bfloat16 *>(dt);
  a.A = A;
  a.D = D;
  a.y = static_cast<__nv_bfloat16 *>(y);
  a.err = err;
  a.L = (int)d.L;
  a.nh = (int)d.nh;
  a.S = (int)d.S;
  a.hpg = (int)d.hpg;
  a.T = (int)d.T;
  a.nc = (int)d.nc;
  a.nb = (int)d.b;
  a.hs = hs;
  a.off_C = l.off_C;
  a.off_B = l.off_B;
  a.off_hx0 = l.off_hx[0];
  a.off_hx1 = l.off_hx[1];
  const int64_t gy = d.nc * (split ? d.T / 128 : 1);
  if (gy > 65535) return cudaErrorInvalidValue;
  dim3 grid((unsigned)(d.nh / hs), (unsigned)gy, (unsigned)d.b);
  // programmatic stream serialisation, as for fwd_scan: the producer waits
  // on the device before loading the first start state
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, tC, tB, tx, tS, tY, a);
}

}  // namespace ssd
