// Forward path, chunk jump terms (bf16 I/O): for every chunk k and head h,
//
//   dH[k] = sum_{j in chunk} (exp2(G_last - G_j) dt_j) B_j (outer) x_j      (S x P)
//   gamma[k] = (exp2(G_last), the scale of the stored start state)
//
// ("Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA
// CUDA Tile", section "Mamba-2 architecture": the second term of the
// log-space jump h_{t+T} = exp(G_last) h_t + (exp(G_last - G) B)^T X, with the
// in-chunk cumsum G of "Kernel 1" computed here.)  All chunks are
// independent, so this runs fully in parallel; the sequential part is the
// bandwidth kernel in fwd_state_pass.cu.
//
// Persistent: one or two CTAs per SM (the launch plan) walk a strided list
// of work items, an item being (chunk, S slice, group of H heads that share
// B, batch); an S slice is 128 rows of S, or both halves of S when S > 128
// (kNsl = 2: x is then scaled once for the two M = 128 accumulations).
// The shared-memory ring of 64-token blocks runs across item boundaries, and
// the tensor-memory accumulators are double-buffered by item, so the loads
// of item j+1 stream in while item j is reduced and item j-1 is written out.
// Warp roles:
//   warp 8 (TMA):  per block, B (MN-major, s contiguous; once for the H heads)
//                  and x of each head (MN-major);
//   warp 9 (MMA):  per block and slice, M = 128 (s) x N = H P MMAs (one per
//                  head when P is not a multiple of 64) into the item's
//                  accumulator set (lane = s, column = (slice H + head) P + p);
//   warps 0-7:     per item, the heads' in-chunk cumsums and jump weights
//                  (dt and A fetched one item ahead), the scaling of each x
//                  row by its weight in shared memory, then the previous
//                  item's epilogue (with one CTA per SM and kNsl = 2 spread
//                  over the item's stages): each dH tile staged in shared
//                  memory and written by a TMA store as bf16
//                  [b, nh, nc, S, P] (p contiguous, the layout the output
//                  kernel reads); gamma as fp32 pairs (decay, state
//                  scale: 2^alpha with the factored output pass, else 1).
// With the factored output pass (fwd_out.cu) selected, the row warps also
// write what that pass needs of each chunk's in-chunk cumsum G: the anchor
// alpha (the integer nearest G_last / 2) and whether the chunk is too steep
// for the factored decay, and per token u = exp2(G - alpha) and
// v = exp2(alpha - G) dt, all in fp32.
#include "fwd.cuh"

namespace ssd {
namespace {

constexpr int kRowWarps = 8;
constexpr int kRowThreads = kRowWarps * 32;
constexpr int kThreads = kRowThreads + 64;
constexpr int kProducerWarp = kRowWarps, kMmaWarp = kRowWarps + 1;
constexpr int kKB = 64;     // tokens per pipeline stage
constexpr int kMaxNST = 4;  // pipeline stages (at most)
constexpr int kBlk = kKB * 128;   // 64 rows of 128 bytes
constexpr int kOutBlk = 128 * 128;  // one staged dH tile: 128 s rows x 64 p
// Range limits of the factored decay of the output pass (fwd_out.cu): the
// largest total decay of a chunk (log2 units), and the smallest column factor
// of a real token.
constexpr float kSpanMax = 180.f;
constexpr float kMinFactor = 7.52316384526264e-37f;  // 2^-120

struct CsArgs {
  const __nv_bfloat16 *dt;
  const float *A;
  float2 *gamma;
  // factored-decay outputs (all null unless the output pass wants them):
  // u, v [b, nh, nc * T]; anchor [b, nh, nc] = (alpha, steep ? 1 : 0)
  float *u, *v;
  float2 *anchor;
  int *err;
  int L, nh, P, S, hpg, T, nc, H, n_st, n_hg, nst, n_items, nout;
  int nb;  // batch count (the extents the debug-bounds checks use)
};

// Work item -> (batch, chunk, S slice, first head).  The head groups of one
// (chunk, slice) are adjacent, so CTAs running at the same time share B in L2.
struct Item {
  int b, k, st, hbase;
};
__device__ __forceinline__ Item decode(int item, const CsArgs &a) {
  Item it;
  const int hg = item % a.n_hg;
  int r = item / a.n_hg;
  it.st = r % a.n_st;
  r /= a.n_st;
  it.k = r % a.nc;
  it.b = r / a.nc;
  it.hbase = hg * a.H;
  return it;
}

// kCtas CTAs per SM: 1 (items of up to 4 heads, H P <= 256) or 2 (up to 2
// heads, H P <= 128, so that two CTAs share the tensor memory).
template <int kCtas, int kNsl>
__global__ void __launch_bounds__(kThreads, kCtas)
fwd_chunk_state_bf16(const __grid_constant__ CUtensorMap tm_B,
                     const __grid_constant__ CUtensorMap tm_x,
                     const __grid_constant__ CUtensorMap tm_dH, const CsArgs a) {
  constexpr int kMaxH = kCtas == 1 ? 4 : 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full[kMaxNST], scaled[kMaxNST], empty[kMaxNST], acc_full[2],
      acc_free[2];
  __shared__ uint32_t tmem_slot;
  __shared__ float w_s[2][kMaxH][256];             // jump weights, by item parity
  __shared__ float warp_tot[2][kMaxH][kRowWarps];  // cumsum partials, by item parity
  __shared__ int warp_fok[2][kMaxH][kRowWarps];    // factored-decay range checks

  const int L = a.L, nh = a.nh, P = a.P, T = a.T, nc = a.nc, H = a.H, nst = a.nst;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int nPb = (P + 63) / 64;
  const int xbytes = nPb * kBlk;                  // one head's x block
  constexpr int nsl = kNsl;
  const int stage_bytes = 2 * nsl * kBlk + H * xbytes;  // B blocks | x blocks
  uint8_t *ostage = smem + nst * stage_bytes;     // a.nout staged dH tiles
  const int obytes = nPb * kOutBlk;
  const int HP = H * P;
  // accumulator set (item parity) `set`, S slice sl, head q: columns
  // (set nsl + sl) H P + q P
  const int acc_cols = nsl * HP;
  const uint32_t ncols = 2 * acc_cols <= 32    ? 32
                         : 2 * acc_cols <= 64  ? 64
                         : 2 * acc_cols <= 128 ? 128
                         : 2 * acc_cols <= 256 ? 256
                                               : 512;

  if (tid == 0) {
    for (int i = 0; i < nst; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&scaled[i], kRowThreads);
      ptx::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&acc_full[i], 1);
      ptx::mbar_init(&acc_free[i], kRowThreads);
    }
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
  ptx::griddep_launch_dependents();  // the state pass may be scheduled now

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (leader) {
      ptx::prefetch_tmap(&tm_B);
      ptx::prefetch_tmap(&tm_x);
    }
    int u = 0;
    for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
      const Item it = decode(item, a);
      const int tok0 = it.k * T;
      const int nkb = (min(T, L - tok0) + kKB - 1) / kKB;
      const int g = it.hbase / a.hpg;  // the heads' group: B[b, t, g, :]
      for (int kb = 0; kb < nkb; ++kb, ++u) {
        const int s = u % nst;
        ptx::mbar_wait(&empty[s], ((u / nst) & 1) ^ 1, a.err, 101);
        if (leader) {
          uint8_t *Bb = smem + s * stage_bytes;
          uint8_t *Xb = Bb + 2 * nsl * kBlk;
          const int tok = tok0 + kb * kKB;
          ptx::mbar_arrive_expect_tx(&full[s], stage_bytes);
          for (int mb = 0; mb < 2 * nsl; ++mb)
            ptx::tma_load_4d(Bb + mb * kBlk, &tm_B, it.st * nsl * 128 + mb * 64, g, tok, it.b,
                             &full[s]);
          for (int q = 0; q < H; ++q)
            for (int pb = 0; pb < nPb; ++pb)
              ptx::tma_load_4d(Xb + q * xbytes + pb * kBlk, &tm_x, pb * 64, it.hbase + q, tok,
                               it.b, &full[s]);
        }
        __syncwarp();
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // With P a multiple of 64 the heads' x blocks abut in shared memory and
    // form one N = H P operand: one MMA per K step reads the B tile once.
    const bool merged = (P % 64) == 0;
    const uint32_t idesc = ptx::idesc_bf16(128, merged ? HP : P, true, true);
    const int n_mma = merged ? 1 : H;
    int u = 0, jl = 0;
    for (int item = blockIdx.x; item < a.n_items; item += gridDim.x, ++jl) {
      const Item it = decode(item, a);
      const int nkb = (min(T, L - it.k * T) + kKB - 1) / kKB;
      const int set = jl & 1;
      ptx::mbar_wait(&acc_free[set], ((jl >> 1) & 1) ^ 1, a.err, 102);
      ptx::tc_fence_after();
      for (int kb = 0; kb < nkb; ++kb, ++u) {
        const int s = u % nst;
        ptx::mbar_wait(&scaled[s], (u / nst) & 1, a.err, 103);
        ptx::tc_fence_after();
        if (leader) {
          const uint32_t bs = ptx::smem_u32(smem + s * stage_bytes);
          const uint32_t x0 = bs + 2 * nsl * kBlk;
          for (int sl = 0; sl < nsl; ++sl) {
            const uint32_t b0 = bs + sl * 2 * kBlk;
            for (int q = 0; q < n_mma; ++q) {
#pragma unroll
              for (int kk = 0; kk < kKB / 16; ++kk) {
                const uint64_t ad = ptx::smem_desc(b0 + kk * 2048, kBlk, 1024, ptx::kSw128);
                const uint64_t bd =
                    ptx::smem_desc(x0 + q * xbytes + kk * 2048, kBlk, 1024, ptx::kSw128);
                ptx::mma_ss<false>(tmem + (set * nsl + sl) * HP + q * P, ad, bd, idesc,
                                   (kb | kk) ? 1u : 0u);
              }
            }
          }
          ptx::mma_commit(&empty[s]);
        }
        __syncwarp();
      }
      if (leader) ptx::mma_commit(&acc_full[set]);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ row warps
    const int quad = warp & 3, half = warp >> 2;  // TMEM lane quadrant, column half
    const int lrow = quad * 32 + (tid & 31);       // row of the S slice = TMEM lane
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const int ngrp = P / 16;                       // 16-column groups of a head

    // dt and A of the next item, one token per thread.  dt stays in its
    // bf16 bits until the cumsum uses it, so no instruction waits on the
    // loads before then.
    unsigned short draw[kMaxH];
    float Aq[kMaxH];
    auto fetch = [&](int item) {
#pragma unroll
      for (int q = 0; q < kMaxH; ++q) {
        draw[q] = 0;
        Aq[q] = 0.f;
      }
      if (item >= a.n_items) return;
      const Item it = decode(item, a);
      const int tok0 = it.k * T, valid = min(T, L - tok0);
      const unsigned short *dtp = reinterpret_cast<const unsigned short *>(a.dt);
#pragma unroll
      for (int q = 0; q < kMaxH; ++q)
        if (q < H && SSD_IN_BOUNDS(it.hbase + q < nh && it.b < a.nb, a.err, 40)) {
          Aq[q] = a.A[it.hbase + q];
          if (tid < valid) draw[q] = dtp[((int64_t)it.b * L + tok0 + tid) * nh + it.hbase + q];
        }
    };

    int n_out = 0;  // dH tiles staged so far; tile n uses staging buffer n & 1
    // The epilogue of item jl writes its nsl * H dH tiles, one call of
    // epi_tile per tile: the first waits for the item's accumulators, the
    // last releases them.  With one CTA per SM and two slices of S per item
    // the calls are spread over the next item's x scaling, so that the loads
    // of its later stages arrive meanwhile.
    // one dH tile (S slice sl, head q) of an item with accumulator set `set`
    auto write_tile = [&](const Item &it, int set, int sl, int q) {
      {
        const uint32_t acc = tmem + lane_base + (set * nsl + sl) * HP + q * P;
        uint8_t *stg = ostage + (n_out % a.nout) * obytes;
        // the store that last used this buffer has finished reading it
        if (tid == 0 && n_out >= a.nout) {
          if (a.nout == 2)
            ptx::bulk_wait_read<1>();
          else
            ptx::bulk_wait_read<0>();
        }
        ptx::named_bar_sync(2, kRowThreads);
        for (int g0 = half; g0 < ngrp; g0 += 4) {
          // up to two 16-column groups per pass: g0 and g0 + 2
          uint32_t r0[16], r1[16];
          const bool two = g0 + 2 < ngrp;
          ptx::tmem_ld16(acc + g0 * 16, r0);
          if (two) ptx::tmem_ld16(acc + (g0 + 2) * 16, r1);
          ptx::tmem_ld_wait();
          ptx::reg_fence(r0);
          ptx::reg_fence(r1);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (t == 1 && !two) break;
            const int gg = g0 + 2 * t;
            const uint32_t *r = t ? r1 : r0;
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
            uint8_t *blk = stg + (gg >> 2) * kOutBlk;
#pragma unroll
            for (int e = 0; e < 2; ++e)
              *reinterpret_cast<uint4 *>(blk + sw128(lrow, ((gg & 3) * 2 + e) * 16)) =
                  pack_io16(v + 8 * e, (__nv_bfloat16 *)nullptr);
          }
        }
        ptx::fence_async_smem();
        ptx::named_bar_sync(2, kRowThreads);
        if (tid == 0) {
          const int row3 = ((it.b * nh + it.hbase + q) * nc + it.k);
          for (int pb = 0; pb < nPb; ++pb)
            ptx::tma_store_3d(&tm_dH, stg + pb * kOutBlk, pb * 64, (it.st * nsl + sl) * 128,
                              row3);
          ptx::bulk_commit();
        }
        ++n_out;
      }
    };
    auto epi_tile = [&](const Item &it, int jl, int tile) {
      const int set = jl & 1;
      if (tile == 0) {
        ptx::mbar_wait(&acc_full[set], (jl >> 1) & 1, a.err, 104);
        ptx::tc_fence_after();
      }
      write_tile(it, set, tile / H, tile % H);
      if (tile == nsl * H - 1) {
        ptx::tc_fence_before();
        ptx::mbar_arrive(&acc_free[set]);
      }
    };
    // the whole epilogue of item jl at once
    auto epilogue = [&](const Item &it, int jl) {
      const int set = jl & 1;
      ptx::mbar_wait(&acc_full[set], (jl >> 1) & 1, a.err, 104);
      ptx::tc_fence_after();
      for (int sl = 0; sl < nsl; ++sl)
        for (int q = 0; q < H; ++q) write_tile(it, set, sl, q);
      ptx::tc_fence_before();
      ptx::mbar_arrive(&acc_free[set]);
    };
    constexpr bool kInterleave = kCtas == 1 && kNsl == 2;
    const int n_tiles = nsl * H;

    fetch(blockIdx.x);
    Item prev{0, 0, 0, 0};
    int u = 0, jl = 0;
    for (int item = blockIdx.x; item < a.n_items; item += gridDim.x, ++jl) {
      const Item it = decode(item, a);
      const int tok0 = it.k * T, valid = min(T, L - tok0);
      const int nkb = (valid + kKB - 1) / kKB;
      float(*w)[256] = w_s[jl & 1];
      float(*wt)[kRowWarps] = warp_tot[jl & 1];
      // in-chunk cumsums of the H heads (one token per thread) and the jump
      // weights; the last real token is the last nonzero contribution, so
      // the block total equals G at position valid - 1
      float incl[kMaxH], d[kMaxH];
#pragma unroll
      for (int q = 0; q < kMaxH; ++q) {
        d[q] = __uint_as_float((uint32_t)draw[q] << 16);  // bf16 -> fp32, exact
        incl[q] = Aq[q] * kLog2e * d[q];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float o = __shfl_up_sync(0xffffffffu, incl[q], off);
          if ((tid & 31) >= off) incl[q] += o;
        }
        if ((tid & 31) == 31 && q < H) wt[q][warp] = incl[q];
      }
      ptx::named_bar_sync(1, kRowThreads);
#pragma unroll
      for (int q = 0; q < kMaxH; ++q) {
        if (q >= H) break;
        float base = 0.f, tot = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kRowWarps; ++w2) {
          const float t = wt[q][w2];
          tot += t;
          if (w2 < warp) base += t;
        }
        if (tid < T) w[q][tid] = tid < valid ? exp2f(tot - (base + incl[q])) * d[q] : 0.f;
        if (a.anchor && it.st == 0) {
          // the factors of the output pass about alpha; a real token's
          // column factor must stay a normal bf16 number
          const float Gj = base + incl[q], alpha = rintf(0.5f * tot);
          const float vj = d[q] > 0.f ? ptx::ex2_approx(alpha - Gj) * d[q] : 0.f;
          const bool ok = d[q] == 0.f || vj >= kMinFactor;
          const int all_ok = __all_sync(0xffffffffu, ok);
          if ((tid & 31) == 0) warp_fok[jl & 1][q][warp] = all_ok;
          const int64_t o = ((int64_t)it.b * nh + it.hbase + q) * nc * T + (int64_t)it.k * T + tid;
          if (tid < T && SSD_IN_BOUNDS(o < (int64_t)a.nb * nh * nc * T, a.err, 41)) {
            a.u[o] = ptx::ex2_approx(Gj - alpha);
            a.v[o] = vj;
          }
        }
      }
      ptx::named_bar_sync(1, kRowThreads);
      if (it.st == 0 && tid < H) {
        // thread q: head q's decay, and with the factored output pass its
        // anchor, path and start-state scale
        const int q = tid;
        float tot = 0.f;
        int ok = 1;
#pragma unroll
        for (int w2 = 0; w2 < kRowWarps; ++w2) {
          tot += wt[q][w2];
          if (a.anchor) ok &= warp_fok[jl & 1][q][w2];
        }
        const int64_t o = ((int64_t)it.b * nh + it.hbase + q) * nc + it.k;
        const bool o_ok = SSD_IN_BOUNDS(o < (int64_t)a.nb * nh * nc, a.err, 42);
        float scale = 1.f;
        if (a.anchor) {
          const bool steep = !(ok && -tot <= kSpanMax);
          const float alpha = steep ? 0.f : rintf(0.5f * tot);
          if (o_ok) a.anchor[o] = make_float2(alpha, steep ? 1.f : 0.f);
          scale = __int_as_float((127 + (int)alpha) << 23);  // 2^alpha, alpha in [-91, 0]
        }
        if (o_ok) a.gamma[o] = make_float2(exp2f(tot), scale);
      }
      fetch(item + gridDim.x);  // in flight while this item is scaled

      // scale each head's x rows by its weights: thread = (row, quarter of
      // the row's eight 16-byte chunks), every load issued before the math
      const int r = tid & 63, part = tid >> 6;
      const int nqp = H * nPb;  // 64-column x blocks in a stage, <= 4
      int tile = 0;  // dH tiles of the previous item written so far
      for (int kb = 0; kb < nkb; ++kb, ++u) {
        const int s = u % nst;
        uint8_t *Xb = smem + s * stage_bytes + 2 * nsl * kBlk;
        ptx::mbar_wait(&full[s], (u / nst) & 1, a.err, 105);
        uint4 buf[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if ((i >> 1) < nqp)
            buf[i] = *reinterpret_cast<const uint4 *>(Xb + (i >> 1) * kBlk +
                                                      sw128(r, (part * 2 + (i & 1)) * 16));
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if ((i >> 1) < nqp) {
            const float ws = w[(i >> 1) / nPb][kb * kKB + r];
            float v[8];
            unpack16(buf[i], v, (__nv_bfloat16 *)nullptr);
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] *= ws;
            *reinterpret_cast<uint4 *>(Xb + (i >> 1) * kBlk +
                                       sw128(r, (part * 2 + (i & 1)) * 16)) =
                pack_op16(v, (__nv_bfloat16 *)nullptr);
          }
        ptx::fence_async_smem();
        ptx::mbar_arrive(&scaled[s]);
        // one dH tile of the previous item per stage (tiles per item, up to
        // 4, and stages per item, 4 for a full chunk of 256, mostly match).
        // Only for one CTA per SM with two slices of S per item, where the
        // epilogue is longest: measured 141 -> 131 us on the long-context
        // layer, and 0.5 us slower on items of one slice.  Two CTAs per SM
        // keep the epilogue after the loop (96 registers do not hold both,
        // and the other CTA overlaps it anyway).
        if (kInterleave && jl > 0 && tile < n_tiles) epi_tile(prev, jl - 1, tile++);
      }
      if (jl > 0) {
        if (kInterleave)
          while (tile < n_tiles) epi_tile(prev, jl - 1, tile++);
        else
          epilogue(prev, jl - 1);
      }
      prev = it;
    }
    if (jl > 0) epilogue(prev, jl - 1);
    if (tid == 0) ptx::bulk_wait<0>();  // every dH store complete
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, ncols);
}

// 128-row slices of S per item: both slices when S > 128 (the heads' x is
// scaled once for the two), else one.
int cs_slices(const Dims &d) { return d.S > 128 ? 2 : 1; }

// Heads per item and CTAs per SM.  For each mode (one CTA per SM with up to
// 4 heads, or two with up to 2; the two accumulator sets, 2 nsl H P columns,
// of every resident CTA fitting the 512 tensor-memory columns) H is the
// divisor of the heads per group minimising the bytes the busiest CTA loads
// (items per CTA, rounded up, times B's slices plus H heads of x per item).
// Two CTAs per SM overlap one CTA's cumsum and epilogue with the other's
// loads and MMAs, which pays once each CTA has several items (3 or more) and
// an item holds one slice of S; otherwise one CTA with larger items is
// faster (measured: the long-context layer's chunk-jump kernel takes 141 us
// with one CTA and two heads per item, 151 us with two CTAs and one head).
}  // namespace

CsPlan chunk_state_plan(const Dims &d) {
  const int nsl = cs_slices(d);
  const int64_t n_st = (d.S + 128 * nsl - 1) / (128 * nsl);
  const int64_t sms = sm_count();
  const int nPb = (int)((d.P + 63) / 64);
  auto best_h = [&](int ctas, int hmax, int64_t cols, int64_t *items_out) {
    int best = 1;
    double best_cost = 1e300;
    for (int h = 1; h <= hmax; ++h) {
      if (d.hpg % h || nsl * h * d.P > cols || h * nPb > 4) continue;
      const int64_t items = d.b * d.nc * n_st * (d.nh / h);
      const double per_item = 2.0 * nsl * kBlk + h * nPb * (double)kBlk;
      const double cost = (double)((items + ctas * sms - 1) / (ctas * sms)) * per_item;
      if (cost < best_cost * 0.999) {
        best_cost = cost;
        best = h;
      }
    }
    *items_out = d.b * d.nc * n_st * (d.nh / best);
    return best;
  };
  int64_t items2 = 0, items1 = 0;
  const int h2 = best_h(2, 2, 128, &items2);
  // with two slices of S per item, two CTAs per SM leave one head per item
  // (B loaded once per head): one CTA with two heads per item is faster
  if (nsl == 1 && items2 >= 3 * 2 * sms) return CsPlan{h2, 2};
  const int h1 = best_h(1, 4, 256, &items1);
  return CsPlan{h1, 1};
}

namespace {

// Shared-memory plan of a launch: ring stages and staged output tiles, or
// nst < 2 when the plan does not fit.
struct CsSmem {
  int stage_bytes, nout, nst, smem;
};
CsSmem cs_smem(const Dims &d, const CsPlan &plan) {
  const int nPb = (int)((d.P + 63) / 64);
  CsSmem m;
  m.stage_bytes = 2 * cs_slices(d) * kBlk + plan.H * nPb * kBlk;
  // dynamic shared memory (1 KB of it alignment slack) within 208 KB for
  // one CTA per SM, 104 KB each for two; two staged dH tiles when they fit,
  // else one
  const int budget = (plan.ctas == 1 ? 207 : 103) * 1024;
  const int out1 = nPb * kOutBlk;
  m.nout = (2 * m.stage_bytes + 2 * out1 <= budget) ? 2 : 1;
  m.nst = std::min(kMaxNST, (budget - m.nout * out1) / m.stage_bytes);
  m.smem = m.nst * m.stage_bytes + m.nout * out1 + 1024;
  return m;
}

}  // namespace

bool chunk_state_plan_ok(const Dims &d, const CsPlan &plan) {
  if (d.T > kRowThreads || (plan.ctas != 1 && plan.ctas != 2)) return false;
  const int nPb = (int)((d.P + 63) / 64);
  const int hmax = plan.ctas == 1 ? 4 : 2;
  const int64_t cols = plan.ctas == 1 ? 256 : 128;
  if (plan.H < 1 || plan.H > hmax || d.hpg % plan.H || cs_slices(d) * plan.H * d.P > cols ||
      plan.H * nPb > 4)
    return false;
  return cs_smem(d, plan).nst >= 2;
}

cudaError_t launch_fwd_chunk_state(const Dims &d, const void *x, const void *B, const void *dt,
                                   const float *A, void *dH, float2 *gamma, float *u, float *v,
                                   float2 *anchor, const CsPlan &plan, int *err,
                                   cudaStream_t st) {
  if (!chunk_state_plan_ok(d, plan)) return cudaErrorInvalidValue;
  const int H = plan.H;
  CUtensorMap tB, tx, tD;
  if (!make_tmap_bl(&tB, B, true, d.b, d.L, d.ng, d.S, kKB) ||
      !make_tmap_bl(&tx, x, true, d.b, d.L, d.nh, d.P, kKB))
    return cudaErrorInvalidValue;
  {
    // dH as [b * nh * nc][S][P]; one box = 128 rows of S x 64 columns of P
    const uint64_t dims[3] = {(uint64_t)d.P, (uint64_t)d.S, (uint64_t)(d.b * d.nh * d.nc)};
    const uint64_t strides[2] = {(uint64_t)d.P * 2, (uint64_t)(d.S * d.P * 2)};
    const uint32_t box[3] = {64u, 128u, 1u};
    if (!make_tmap_sw128(&tD, dH, true, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  const CsSmem m = cs_smem(d, plan);
  const int nst = m.nst, nout = m.nout, smem = m.smem;
  // kNsl: 128-row slices of S per item (2 when S > 128: the heads' x is
  // scaled once for both; n_st then counts items along S)
  const int nsl = cs_slices(d);
  auto kernel = plan.ctas == 1 ? (nsl == 1 ? fwd_chunk_state_bf16<1, 1> : fwd_chunk_state_bf16<1, 2>)
                               : (nsl == 1 ? fwd_chunk_state_bf16<2, 1> : fwd_chunk_state_bf16<2, 2>);
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  CsArgs a;
  a.dt = static_cast<const __nv_bfloat16 *>(dt);
  a.A = A;
  a.gamma = gamma;
  a.u = u;
  a.v = v;
  a.anchor = anchor;
  a.err = err;
  a.L = (int)d.L;
  a.nh = (int)d.nh;
  a.P = (int)d.P;
  a.S = (int)d.S;
  a.hpg = (int)d.hpg;
  a.T = (int)d.T;
  a.nc = (int)d.nc;
  a.nb = (int)d.b;
  a.H = H;
  a.n_st = (int)((d.S + 128 * nsl - 1) / (128 * nsl));
  a.n_hg = (int)(d.nh / H);
  a.nst = nst;
  a.nout = nout;
  const int64_t n_items = d.b * d.nc * a.n_st * a.n_hg;
  if (n_items > 0x7fffffffLL || d.b * d.nh * d.nc > 0x7fffffffLL) return cudaErrorInvalidValue;
  a.n_items = (int)n_items;
  const int grid = (int)std::min<int64_t>(n_items, plan.ctas * (int64_t)sm_count());
  kernel<<<grid, kThreads, smem, st>>>(tB, tx, tD, a);
  return cudaGetLastError();
}

}  // namespace ssd
