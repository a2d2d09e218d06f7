// Backward pass: its GEMM-shaped products on the tensor cores in split TF32
// (fp32-grade products on kind::tf32 MMAs).
//
// The adjoint of the chunked recurrence ("State Space Duality (Mamba-2)
// Part III: The Algorithm", section "The SSD algorithm": the chunk states
// h_k enter the outputs of chunk k through C_t h_k and are built from the
// chunk's dt_t exp2(G_last - G_t) x_t B_t^T; the adjoint states R_k =
// dL/dh_{k+1} from exp2(G_s) gy_s c_s^T) needs, per chunk k and group g,
// with x~_t = dt_t exp2(G_last - G_t) x_t and g~y_t = exp2(G_t) gy_t:
//
//   mode 2, the chunks' jump terms (per head h of the group):
//     dH[h][p][s] = sum_t x~_t[(h,p)] B_t[s]      (forward states)
//     dR[h][p][s] = sum_t g~y_t[(h,p)] c_t[s]     (adjoint states)
//   mode 0, before the per-token kernel (rows (h, p) of the group's heads):
//     dxS[t][(h,p)] = sum_s B_t[s] R_k[(h,p)][s],  ysmS[t][(h,p)] = sum_s c_t[s] h_k[(h,p)][s]
//   mode 1, after it:
//     dB_t[s] += sum_(h,p) x~_t[(h,p)] R_k[(h,p)][s],  dC_t[s] += sum_(h,p) g~y_t[(h,p)] h_k[(h,p)][s]
//   mode 3, the in-chunk scores the per-token kernel weighs (once per group):
//     Kcb[i][j] = c_i . B_j for the 128 x 128 token tiles on or below the
//     chunk's diagonal
//
// (the per-token kernel applies the factors dt_t exp2(G_last - G_t) and
// exp2(G_t) of dxS and ysmS as it reads them).
//
// Precision.  A TF32 product keeps 11 bits of each operand, which puts the
// gradient of A off by up to 1.6 % (its terms cancel over the sequence), so
// every operand a is split into hi = tf32(a) (nearest) and lo = a - hi
// (exact in fp32; the tensor core reads its leading 11 bits) and each
// product is lo_a hi_b + hi_a lo_b + hi_a hi_b, accumulated in fp32 in
// tensor memory: the dropped lo_a lo_b and the truncation of lo leave about
// 2^-21 relative per product, near fp32 (the "3xTF32" split used by fp32
// GEMM libraries on TF32 tensor cores).
//
// Work items (output tiles): (product, batch, chunk, group, M tile, N tile
// of 128 or 64 columns).  M tiles: 128 tokens (modes 0, 1 and 3; with
// chunks shorter than 128 tokens the rows past the chunk are computed and
// not stored) or the rows (h, p) of two heads of the group (mode 2; an odd
// group's last tile repeats its head and stores one).  K runs in slices of
// 32 (one 128-byte row of fp32).  K-major operands (the token rows of modes
// 0, 1 and 3, the states of mode 0) land by TMA as 128-byte swizzled rows;
// the others (the states of mode 1, both operands of mode 2) as 32 x 32
// boxes with K along the rows, transposed by the split.
//
// Persistent, one CTA per SM (448 threads, 225 KB of shared memory at N
// tiles of 128): a producer warp streams the slices of the CTA's tiles
// through a five-stage TMA ring; eight split warps read a landed slice
// into registers, split it (hi and lo), hand the stage back and store the
// halves K-major: the token rows' (A) into tensor memory (warp = TMEM lane
// quadrant x half of the slice's K), the other operand's (B) into shared
// memory, each in one of two operand sets; one warp issues per slice
// 3 x 4 MMAs (M = 128, N, K = 8; A from tensor memory) into the tile's
// accumulator (two in tensor memory, by tile parity) and commits them,
// freeing the operand set; four warps read each finished accumulator (warp
// = TMEM lane quadrant) and store, or add into dB / dC.  Every wait is
// bounded.
#include "tc_common.cuh"

namespace ssd {
namespace {

constexpr int kGM = 128;            // MMA M: tokens (modes 0, 1) or rows (h, p) (mode 2)
constexpr int kASlice = kGM * 128;  // bytes of an M x 32 slice (16 KB)
constexpr int kPh = 64;             // headdim

struct GemmArgs {
  float *out[2];
  int *err;
  int L, nh, ng, hpg, S, T, nc, nb, nmt, nnt, nk, n_items;
};

// hi = tf32(a) (nearest), lo = a - hi (exact) of four values
__device__ __forceinline__ void split4(const float4 v, uint4 &hi, uint4 &lo) {
  hi = make_uint4(to_tf32(v.x), to_tf32(v.y), to_tf32(v.z), to_tf32(v.w));
  lo = make_uint4(__float_as_uint(v.x - __uint_as_float(hi.x)),
                  __float_as_uint(v.y - __uint_as_float(hi.y)),
                  __float_as_uint(v.z - __uint_as_float(hi.z)),
                  __float_as_uint(v.w - __uint_as_float(hi.w)));
}

constexpr int kRowWarps = 8;                  // split warps 0..7
constexpr int kRowThreads = 32 * kRowWarps;
constexpr int kProdWarp = 8, kMmaWarp = 9;    // TMA producer, MMA issuer
constexpr int kEpiWarp0 = 10;                 // epilogue warps 10..13
constexpr int kPThreads = 32 * (kEpiWarp0 + 4);
constexpr int kRing = 5;                      // TMA landing stages

// A landed K-major slice of kBytes: this thread's 16-byte pieces tid + 256 i
// into registers ...
template <int kBytes>
__device__ __forceinline__ void k_read(const uint8_t *buf, int tid,
                                       float4 (&v)[kBytes / 16 / kRowThreads]) {
#pragma unroll
  for (int i = 0; i < kBytes / 16 / kRowThreads; ++i)
    v[i] = *reinterpret_cast<const float4 *>(buf + 16 * (tid + i * kRowThreads));
}
// ... split in registers ...
template <int kN4>
__device__ __forceinline__ void split_regs(const float4 (&v)[kN4], uint4 (&h)[kN4],
                                           uint4 (&l)[kN4]) {
#pragma unroll
  for (int i = 0; i < kN4; ++i) split4(v[i], h[i], l[i]);
}
// ... and stored: hi and lo at the same offsets of their buffers
template <int kBytes>
__device__ __forceinline__ void k_store(uint8_t *hi, uint8_t *lo, int tid,
                                        const uint4 (&h)[kBytes / 16 / kRowThreads],
                                        const uint4 (&l)[kBytes / 16 / kRowThreads]) {
#pragma unroll
  for (int i = 0; i < kBytes / 16 / kRowThreads; ++i) {
    const int off = 16 * (tid + i * kRowThreads);
    *reinterpret_cast<uint4 *>(hi + off) = h[i];
    *reinterpret_cast<uint4 *>(lo + off) = l[i];
  }
}

// A slice that landed as kBoxes boxes of 32 (K) x 32 (M or N) fp32: box j,
// row = K index, 16-byte piece c = M/N indices 32 j + 4 c .. + 3.  Warp w
// takes pieces w, w + 8, ... of the 8 kBoxes pieces per row, lane = row.
template <int kBoxes>
__device__ __forceinline__ void t_read(const uint8_t *buf, int warp, int lane,
                                       float4 (&v)[kBoxes]) {
#pragma unroll
  for (int i = 0; i < kBoxes; ++i) {
    const int idx = warp + 8 * i, j = idx >> 3, c = idx & 7;
    v[i] = *reinterpret_cast<const float4 *>(buf + j * 4096 + sw128(lane, 16 * c));
  }
}
// ... and, split, stored K-major: row 32 j + 4 c + e (an M or N index), K
// index = lane, hi and lo into their buffers
template <int kBoxes>
__device__ __forceinline__ void t_store(uint8_t *hi, uint8_t *lo, int warp, int lane,
                                        const uint4 (&h)[kBoxes], const uint4 (&l)[kBoxes]) {
#pragma unroll
  for (int i = 0; i < kBoxes; ++i) {
    const int idx = warp + 8 * i, j = idx >> 3, c = idx & 7;
    const uint32_t h4[4] = {h[i].x, h[i].y, h[i].z, h[i].w};
    const uint32_t l4[4] = {l[i].x, l[i].y, l[i].z, l[i].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t o = sw128(32 * j + 4 * c + e, 4 * lane);
      *reinterpret_cast<uint32_t *>(hi + o) = h4[e];
      *reinterpret_cast<uint32_t *>(lo + o) = l4[e];
    }
  }
}

// A work item (one output tile): product, batch, chunk, group, M tile, N
// tile, N fastest (CTAs in flight share their operands in L2).
struct Tile {
  int nt, mt, g, k, b, which, mi, ni, tok0, valid, nk;
};
template <int kMode>
__device__ __forceinline__ Tile decode_tile(int item, const GemmArgs &a) {
  Tile t;
  int r = item;
  t.nt = r % a.nnt;
  r /= a.nnt;
  t.mt = r % a.nmt;
  r /= a.nmt;
  t.g = r % a.ng;
  r /= a.ng;
  t.k = r % a.nc;
  r /= a.nc;
  t.b = r % a.nb;
  t.which = r / a.nb;
  // mode 3: the row and column token tiles (mi, ni), ni <= mi, of pair mt
  t.mi = 0;
  t.ni = t.mt;
  if (kMode == 3)
    while (t.ni > t.mi) t.ni -= ++t.mi;
  t.tok0 = t.k * a.T;
  t.valid = min(a.T, a.L - t.tok0);
  t.nk = kMode == 2 ? (t.valid + 31) / 32 : a.nk;
  return t;
}

// Persistent: one CTA per SM walks a strided list of tiles; the slices of
// consecutive tiles stream through one pipeline.  Warp roles:
//   warp 8 (TMA):       slices into a ring of kRing landing stages;
//   warps 0-7 (split):  a landed slice into registers (the stage is then
//                       free), split into hi and lo, written K-major into
//                       one of two operand sets;
//   warp 9 (MMA):       per slice 3 x 4 MMAs from an operand set into the
//                       tile's accumulator (two in tensor memory, by tile
//                       parity), each commit freeing the set;
//   warps 10-13:        per tile the epilogue of its accumulator (warp =
//                       TMEM lane quadrant), which it then frees.
template <int kMode, int kN>
__global__ void __launch_bounds__(kPThreads, 1)
bwd_state_gemm_kernel(const __grid_constant__ CUtensorMap tA0,
                      const __grid_constant__ CUtensorMap tA1,
                      const __grid_constant__ CUtensorMap tS0,
                      const __grid_constant__ CUtensorMap tS1, const GemmArgs a) {
  constexpr bool kTransA = kMode == 2, kTransB = kMode == 1 || kMode == 2;
  constexpr int kBSlice = kN * 128;           // bytes of an N x 32 slice
  constexpr int kStage = kASlice + kBSlice;   // one landed slice
  constexpr int kOps = 2 * kBSlice;           // operand set in smem: hi B | lo B
  // tensor memory: two accumulators (kN columns each), then two operand
  // sets of A (hi in 32 columns, lo in the next 32)
  constexpr int kAcol = 2 * kN;
  constexpr int kTmemCols = kAcol + 128 <= 256 ? 256 : 512;
  constexpr int kNB = kBSlice / 16 / kRowThreads;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *ring = smem, *ops = smem + kRing * kStage;
  // full: a slice landed; empty: the split warps have read it; opfull: an
  // operand set is written; opfree: its MMAs are done; accfull: a tile's
  // MMAs are done; accfree: its epilogue has read the accumulator
  __shared__ __align__(8) uint64_t full[kRing], empty[kRing], opfull[2], opfree[2], accfull[2],
      accfree[2];
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < kRing; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&empty[i], kRowWarps);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&opfull[i], kRowWarps);
      ptx::mbar_init(&opfree[i], 1);
      ptx::mbar_init(&accfull[i], 1);
      ptx::mbar_init(&accfree[i], 4);
    }
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(&tmem_slot, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tA0);
      ptx::prefetch_tmap(&tA1);
      ptx::prefetch_tmap(&tS0);
      ptx::prefetch_tmap(&tS1);
    }
    int u = 0;  // slices issued
    for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
      const Tile t = decode_tile<kMode>(item, a);
      const CUtensorMap *tA = t.which ? &tA1 : &tA0;
      const CUtensorMap *tS = t.which ? &tS1 : &tS0;
      const int t0 = t.tok0 + (kMode == 3 ? t.mi : t.mt) * kGM;
      const int srow = ((t.b * a.nc + t.k) * a.nh + t.g * a.hpg) * kPh;
      const int h0 = t.g * a.hpg + 2 * t.mt;
      const int h1 = h0 + 1 < (t.g + 1) * a.hpg ? h0 + 1 : h0;
      for (int kb = 0; kb < t.nk; ++kb, ++u) {
        const int s = u % kRing, j = u / kRing;
        if (j > 0) ptx::mbar_wait(&empty[s], (j - 1) & 1, a.err, 244);
        if (lane == 0) {
          uint8_t *st = ring + s * kStage;
          uint64_t *bar = &full[s];
          ptx::mbar_arrive_expect_tx(bar, kStage);
          if (kMode == 0) {
            ptx::tma_load_4d(st, tA, 32 * kb, t.g, t0, t.b, bar);
            ptx::tma_load_2d(st + kASlice, tS, 32 * kb, srow + t.nt * kN, bar);
          } else if (kMode == 3) {
            ptx::tma_load_4d(st, tA, 32 * kb, t.g, t0, t.b, bar);
            ptx::tma_load_4d(st + kASlice, tS, 32 * kb, t.g, t.tok0 + t.ni * kGM, t.b, bar);
          } else if (kMode == 1) {
            ptx::tma_load_4d(st, tA, 32 * (kb & 1), t.g * a.hpg + (kb >> 1), t0, t.b, bar);
#pragma unroll
            for (int jb = 0; jb < kN / 32; ++jb)
              ptx::tma_load_2d(st + kASlice + jb * 4096, tS, t.nt * kN + 32 * jb, srow + 32 * kb,
                               bar);
          } else {
            const int tk = t.tok0 + 32 * kb;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              ptx::tma_load_4d(st + q * 4096, tA, 32 * (q & 1), q < 2 ? h0 : h1, tk, t.b, bar);
#pragma unroll
            for (int jb = 0; jb < kN / 32; ++jb)
              ptx::tma_load_4d(st + kASlice + jb * 4096, tS, t.nt * kN + 32 * jb, t.g, tk, t.b,
                               bar);
          }
        }
        __syncwarp();
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = ptx::idesc_tf32(kGM, kN, false, false);
    int u = 0, jl = 0;
    for (int item = blockIdx.x; item < a.n_items; item += gridDim.x, ++jl) {
      const Tile t = decode_tile<kMode>(item, a);
      const int acc = jl & 1;
      if (jl >= 2) ptx::mbar_wait(&accfree[acc], ((jl >> 1) - 1) & 1, a.err, 245);
      ptx::tc_fence_after();
      for (int kb = 0; kb < t.nk; ++kb, ++u) {
        const int ob = u & 1;
        ptx::mbar_wait(&opfull[ob], (u >> 1) & 1, a.err, 246);
        ptx::tc_fence_after();
        if (lane == 0) {
          const uint32_t o = ptx::smem_u32(ops + ob * kOps);
          const uint32_t bh = o, bl = o + kBSlice;
          const uint32_t ah = tmem + kAcol + 64 * ob, al = ah + 32;  // A in tensor memory
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t dbh = ptx::smem_desc(bh + 32 * kk, 16, 1024, ptx::kSw128);
            const uint64_t dbl = ptx::smem_desc(bl + 32 * kk, 16, 1024, ptx::kSw128);
            const uint32_t d = tmem + acc * kN;
            ptx::mma_ts_tf32(d, al + 8 * kk, dbh, idesc, (kb | kk) ? 1u : 0u);
            ptx::mma_ts_tf32(d, ah + 8 * kk, dbl, idesc, 1u);
            ptx::mma_ts_tf32(d, ah + 8 * kk, dbh, idesc, 1u);
          }
          ptx::mma_commit(&opfree[ob]);
        }
        __syncwarp();
      }
      if (lane == 0) ptx::mma_commit(&accfull[acc]);
      __syncwarp();
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3, m = quad * 32 + lane;  // TMEM lane quadrant, row
    int jl = 0;
    for (int item = blockIdx.x; item < a.n_items; item += gridDim.x, ++jl) {
      const Tile t = decode_tile<kMode>(item, a);
      const int acc = jl & 1;
      bool live;
      int64_t o_row;  // the element offset of column nt kN of this thread's row
      if (kMode == 2) {
        const int h0 = t.g * a.hpg + 2 * t.mt;
        const int h1 = h0 + 1 < (t.g + 1) * a.hpg ? h0 + 1 : h0;
        const int hl = m >> 6, p = m & (kPh - 1);
        live = hl == 0 || h1 != h0;
        o_row = ((((int64_t)t.b * a.nh + (hl ? h1 : h0)) * a.nc + t.k) * kPh + p) * a.S +
                t.nt * kN;
      } else if (kMode == 3) {
        const int i = t.mi * kGM + m;  // row token of the chunk
        live = i < a.T;
        o_row = (((int64_t)t.b * a.ng + t.g) * a.nc + t.k) * a.T * a.T + (int64_t)i * a.T +
                t.ni * kGM;
      } else {
        const int tl = t.mt * kGM + m;  // chunk-relative token
        live = tl < t.valid;
        const int64_t tok = (int64_t)t.b * a.L + t.tok0 + tl;
        o_row = kMode == 0 ? (tok * a.nh + (int64_t)t.g * a.hpg) * kPh + t.nt * kN
                           : (tok * a.ng + t.g) * a.S + t.nt * kN;
      }
      const int64_t o_end = kMode == 1 ? (int64_t)a.nb * a.L * a.ng * a.S
                          : kMode == 0 ? (int64_t)a.nb * a.L * a.nh * kPh
                          : kMode == 3 ? (int64_t)a.nb * a.ng * a.nc * a.T * a.T
                                       : (int64_t)a.nb * a.nh * a.nc * kPh * a.S;
      (void)o_end;  // read by the debug-bounds checks only
      float *out = t.which ? a.out[1] : a.out[0];
      ptx::mbar_wait(&accfull[acc], (jl >> 1) & 1, a.err, 247);
      ptx::tc_fence_after();
#pragma unroll 2
      for (int c0 = 0; c0 < kN; c0 += 16) {
        float v[16];
        ptx::tmem_ld16_sync(tmem + ((uint32_t)(quad * 32) << 16) + acc * kN + c0, v);
        const int64_t o = o_row + c0;
        if (kMode == 3 && t.ni * kGM + c0 >= a.T) continue;  // columns past the chunk
        if (!live || !SSD_IN_BOUNDS(o + 16 <= o_end, a.err, 243)) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float4 w4 = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          if (kMode == 1) {
            const float4 w = *reinterpret_cast<const float4 *>(out + o + 4 * q);
            w4.x += w.x;
            w4.y += w.y;
            w4.z += w.z;
            w4.w += w.w;
          }
          *reinterpret_cast<float4 *>(out + o + 4 * q) = w4;
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&accfree[acc]);
    }
  } else {
    // ------------------------------------------------------------ split warps
    int u = 0;  // slices consumed
    for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
      const Tile t = decode_tile<kMode>(item, a);
      for (int kb = 0; kb < t.nk; ++kb, ++u) {
        const int s = u % kRing, ob = u & 1;
        ptx::mbar_wait(&full[s], (u / kRing) & 1, a.err, 240);
        const uint8_t *st = ring + s * kStage, *sb = st + kASlice;
        // A: this warp's TMEM lane quadrant q (row m = 32 q + lane) and half
        // kh of the slice's K, 16 values; B: pieces as for a K-major or
        // transposed slice
        const int q = warp & 3, kh = warp >> 2, m = 32 * q + lane;
        float av[16];
        if constexpr (kTransA) {
          // box q holds rows K (tokens) x 32 M-rows: column lane, rows 16 kh ..
#pragma unroll
          for (int e = 0; e < 16; ++e)
            av[e] = *reinterpret_cast<const float *>(st + q * 4096 + sw128(16 * kh + e, 4 * lane));
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float4 v = *reinterpret_cast<const float4 *>(st + sw128(m, 64 * kh + 16 * j));
            av[4 * j] = v.x;
            av[4 * j + 1] = v.y;
            av[4 * j + 2] = v.z;
            av[4 * j + 3] = v.w;
          }
        }
        float4 vb[kNB];
        if constexpr (kTransB) t_read<kNB>(sb, warp, lane, vb);
        else k_read<kBSlice>(sb, tid, vb);
        // split in registers: the loads have returned before the stage is
        // handed back to the TMA (an async-proxy write after these
        // generic-proxy reads, ordered by the proxy fence and the barrier)
        uint32_t ahi[16], alo[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          ahi[e] = to_tf32(av[e]);
          alo[e] = __float_as_uint(av[e] - __uint_as_float(ahi[e]));
        }
        uint4 hb[kNB], lb[kNB];
        split_regs(vb, hb, lb);
        ptx::fence_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&empty[s]);  // the stage may be refilled
        if (u >= 2) ptx::mbar_wait(&opfree[ob], ((u >> 1) - 1) & 1, a.err, 241);
        ptx::tc_fence_after();
        const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + kAcol + 64 * ob + 16 * kh;
        ptx::tmem_st16u(ta, ahi);
        ptx::tmem_st16u(ta + 32, alo);
        uint8_t *o = ops + ob * kOps;
        if constexpr (kTransB) t_store<kNB>(o, o + kBSlice, warp, lane, hb, lb);
        else k_store<kBSlice>(o, o + kBSlice, tid, hb, lb);
        ptx::tmem_st_wait();
        ptx::fence_async_smem();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&opfull[ob]);
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, kTmemCols);
}

template <int kMode, int kN>
cudaError_t run_gemm(const CUtensorMap &ta0, const CUtensorMap &ta1, const CUtensorMap &ts0,
                     const CUtensorMap &ts1, const GemmArgs &a, cudaStream_t st) {
  constexpr int kStage = kASlice + kN * 128;
  constexpr int smem = kRing * kStage + 2 * 2 * kN * 128 + 1024;  // ring, two B operand sets
  auto kernel = bwd_state_gemm_kernel<kMode, kN>;
  const cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = (int)std::min<int64_t>(a.n_items, sm_count());
  kernel<<<grid, kPThreads, smem, st>>>(ta0, ta1, ts0, ts1, a);
  return cudaGetLastError();
}

template <int kMode>
cudaError_t run_mode(int kN, const CUtensorMap &ta0, const CUtensorMap &ta1,
                     const CUtensorMap &ts0, const CUtensorMap &ts1, const GemmArgs &a,
                     cudaStream_t st) {
  return kN == 128 ? run_gemm<kMode, 128>(ta0, ta1, ts0, ts1, a, st)
                   : run_gemm<kMode, 64>(ta0, ta1, ts0, ts1, a, st);
}

}  // namespace

bool bwd_state_gemm_supported(const Dims &d) {
  return d.P == kPh && (d.S == 64 || d.S == 128 || d.S == 256) && d.T >= 32 && d.T % 32 == 0 &&
         d.b * d.nc * d.nh * kPh < (1LL << 31) && d.b * d.L < (1LL << 31);
}

cudaError_t launch_bwd_gemm(const Dims &d, int mode, int nprod, const float *A0, const float *A1,
                            const float *S0, const float *S1, float *out0, float *out1, int *err,
                            cudaStream_t st) {
  if (!bwd_state_gemm_supported(d) || mode < 0 || mode > 3 || nprod < 1 || nprod > 2)
    return cudaErrorInvalidValue;
  if (nprod == 1) {
    A1 = A0;
    S1 = S0;
    out1 = out0;
  }
  const int64_t hp = d.hpg * kPh;
  const int kN = mode == 3 ? 128 : (mode == 0 ? hp : d.S) % 128 == 0 ? 128 : 64;
  CUtensorMap ta0, ta1, ts0, ts1;
  // token-row operands: B, C ([b, L, ng, S]) or x~, gy~ ([b, L, nh, P]), in
  // boxes of 32 columns x 128 tokens (modes 0, 1) or 32 tokens (mode 2)
  const bool a_bc = mode == 0 || mode == 3;
  const int rows = mode == 2 ? 32 : kGM;
  if (!make_tmap_bl(&ta0, A0, false, d.b, d.L, a_bc ? d.ng : d.nh, a_bc ? d.S : kPh, rows) ||
      !make_tmap_bl(&ta1, A1, false, d.b, d.L, a_bc ? d.ng : d.nh, a_bc ? d.S : kPh, rows))
    return cudaErrorInvalidValue;
  if (mode >= 2) {
    // B, C in boxes of 32 s x 32 tokens (mode 2) or 128 tokens (mode 3)
    const int srows = mode == 2 ? 32 : kGM;
    if (!make_tmap_bl(&ts0, S0, false, d.b, d.L, d.ng, d.S, srows) ||
        !make_tmap_bl(&ts1, S1, false, d.b, d.L, d.ng, d.S, srows))
      return cudaErrorInvalidValue;
  } else {
    // the states as a [b nc nh P][S] matrix: boxes of 32 s x (N rows in
    // mode 0, 32 rows in mode 1)
    const uint64_t dims[2] = {(uint64_t)d.S, (uint64_t)(d.b * d.nc * d.nh * kPh)};
    const uint64_t strides[1] = {(uint64_t)d.S * 4};
    const uint32_t box[2] = {32u, mode == 1 ? 32u : (uint32_t)kN};
    if (!make_tmap_sw128(&ts0, S0, false, 2, dims, strides, box) ||
        !make_tmap_sw128(&ts1, S1, false, 2, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  GemmArgs a;
  a.out[0] = out0;
  a.out[1] = out1;
  a.err = err;
  a.L = (int)d.L;
  a.nh = (int)d.nh;
  a.ng = (int)d.ng;
  a.hpg = (int)d.hpg;
  a.S = (int)d.S;
  a.T = (int)d.T;
  a.nc = (int)d.nc;
  a.nb = (int)d.b;
  const int64_t ntok = (d.T + kGM - 1) / kGM;  // 128-token tiles per chunk
  a.nmt = (int)(mode == 2 ? (d.hpg + 1) / 2 : mode == 3 ? ntok * (ntok + 1) / 2 : ntok);
  a.nnt = (int)(mode == 3 ? 1 : (mode == 0 ? hp : d.S) / kN);
  a.nk = (int)(mode == 1 ? 2 * d.hpg : mode == 2 ? 0 : d.S / 32);
  const int64_t n_items = nprod * d.b * d.nc * d.ng * a.nmt * a.nnt;
  if (n_items <= 0 || n_items > 0x7fffffffLL) return cudaErrorInvalidValue;
  a.n_items = (int)n_items;
  switch (mode) {
    case 0:
      return run_mode<0>(kN, ta0, ta1, ts0, ts1, a, st);
    case 1:
      return run_mode<1>(kN, ta0, ta1, ts0, ts1, a, st);
    case 2:
      return run_mode<2>(kN, ta0, ta1, ts0, ts1, a, st);
    default:
      return run_gemm<3, 128>(ta0, ta1, ts0, ts1, a, st);
  }
}

}  // namespace ssd
