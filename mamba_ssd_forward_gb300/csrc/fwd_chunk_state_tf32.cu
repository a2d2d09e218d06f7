// Forward path, chunk jump terms with fp32 I/O (kind::tf32 MMAs): for every
// chunk k and head h,
//
//   dstates[k][p][s] = sum_{j in chunk} w_j x_j[p] B_j[s],   w_j = exp2(G_last - G_j) dt_j
//
// ("Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA
// CUDA Tile", section "Mamba-2 architecture": the second term of the
// log-space jump h_{t+T} = exp(G_last) h_t + (exp(G_last - G) B)^T X, with G
// the in-chunk cumsum of A dt of "Kernel 1", in log2 units, computed here
// and written out for the state pass and the output pass).  The fp32 twin of
// fwd_chunk_state.cu: the same contraction as an M = 128 (s) x N = H P MMA
// over the chunk's tokens, with H heads of one group sharing each load of B.
//
// kind::tf32 takes K-major operands only, and both operands arrive with the
// tokens along the rows (s or p contiguous).  So every landed 32 x 32 box
// is transposed in place by the row warps (each thread reads one 16-byte
// piece of a row, all threads meet at a barrier, then each writes its four
// values down a column), rounding to tf32 and, for x, scaling each token by
// w_j on the way.
//
// Persistent: one CTA per SM walks a strided list of work items (chunk,
// 128-row slice of S, group of H heads, batch); the ring of 32-token stages
// runs across item boundaries and the tensor-memory accumulators are
// double-buffered by item, so item j + 1 streams in while item j is reduced
// and item j - 1 is written out.  Warp roles:
//   warp 8 (TMA):  per stage, B (four boxes of 32 tokens x 32 s) and each
//                  head's x (two boxes of 32 tokens x 32 p);
//   warp 9 (MMA):  per stage four K = 8 steps of D[s][(head, p)] (N = H P,
//                  up to 256) into the item's accumulator set;
//   warps 0-7:     per item the heads' in-chunk cumsums (written to G once,
//                  by the items of the first slice of S) and jump weights,
//                  per stage the in-place
//                  transposition, per item the previous item's epilogue
//                  (thread = s: stores along s are coalesced).
// Supported: P = 64, S a multiple of 64, T in {128, 256} (S = 64 runs as a
// 128-row slice whose upper half reads zeros: TMA fills the boxes past S).
#include "fwd.cuh"

namespace ssd {
namespace {

constexpr int kRowWarps = 8;
constexpr int kRowThreads = kRowWarps * 32;
constexpr int kThreads = kRowThreads + 64;
constexpr int kProducerWarp = kRowWarps, kMmaWarp = kRowWarps + 1;
constexpr int kP = 64;
constexpr int kKB = 32;         // tokens per stage (one K atom of tf32)
constexpr int kBox = 32 * 128;  // one 32 x 32 fp32 box
constexpr int kMaxH = 4;        // heads per item
constexpr int kMaxSt = 8;       // ring stages (at most)

struct CsArgs32 {
  const float *dt, *A;
  float *G;  // in-chunk cumsums out, log2 units, [b, nh, nc * T]
  float *dstates;
  int *err;
  int L, nh, S, hpg, T, nc, nb, H, n_st, n_hg, nst, n_items;
};

struct Item32 {
  int b, k, st, hbase;
};
__device__ __forceinline__ Item32 decode32(int item, const CsArgs32 &a) {
  Item32 it;
  const int hg = item % a.n_hg;
  int r = item / a.n_hg;
  it.st = r % a.n_st;
  r /= a.n_st;
  it.k = r % a.nc;
  it.b = r / a.nc;
  it.hbase = hg * a.H;
  return it;
}

template <int kT>
__global__ void __launch_bounds__(kThreads, 1)
fwd_chunk_state_tf32(const __grid_constant__ CUtensorMap tm_B,
                     const __grid_constant__ CUtensorMap tm_x, const CsArgs32 a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  // full: a stage landed; ready: the row warps transposed it; empty: the
  // MMAs reading it are done
  __shared__ __align__(8) uint64_t full[kMaxSt], ready[kMaxSt], empty[kMaxSt], acc_full[2],
      acc_free[2];
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(16) float ws[2][kMaxH][256];  // jump weights, by item parity
  __shared__ float warp_tot[2][kMaxH][kRowWarps];     // cumsum partials, by item parity

  const int L = a.L, nh = a.nh, S = a.S, H = a.H, nst = a.nst, nc = a.nc;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int HP = H * kP;
  const int stage_bytes = 4 * kBox + H * 2 * kBox;  // B (128 s) | x (H heads)
  auto stage_ptr = [&](int u) { return smem + (u % nst) * stage_bytes; };

  if (tid == 0) {
    for (int i = 0; i < nst; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&ready[i], kRowWarps);
      ptx::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&acc_full[i], 1);
      ptx::mbar_init(&acc_free[i], kRowWarps);
    }
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(&tmem_slot, 2 * HP <= 256 ? 256 : 512);
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
      const Item32 it = decode32(item, a);
      const int tok0 = it.k * kT;
      const int nkb = (min(kT, L - tok0) + kKB - 1) / kKB;
      const int g = it.hbase / a.hpg;
      for (int kb = 0; kb < nkb; ++kb, ++u) {
        const int sl = u % nst;
        ptx::mbar_wait(&empty[sl], ((u / nst) & 1) ^ 1, a.err, 180);
        if (leader) {
          uint8_t *st = stage_ptr(u);
          const int tok = tok0 + kb * kKB;
          ptx::mbar_arrive_expect_tx(&full[sl], stage_bytes);
          for (int i = 0; i < 4; ++i)
            ptx::tma_load_4d(st + i * kBox, &tm_B, it.st * 128 + 32 * i, g, tok, it.b, &full[sl]);
          for (int q = 0; q < H; ++q)
            for (int ph = 0; ph < 2; ++ph)
              ptx::tma_load_4d(st + (4 + 2 * q + ph) * kBox, &tm_x, 32 * ph, it.hbase + q, tok,
                               it.b, &full[sl]);
        }
        __syncwarp();
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // One MMA per K step: A = B^T (128 rows of s), B operand = the H heads'
    // transposed x tiles, which abut in the stage (N = H P).
    const uint32_t idesc = ptx::idesc_tf32(128, HP, false, false);
    int u = 0, jl = 0;
    for (int item = blockIdx.x; item < a.n_items; item += gridDim.x, ++jl) {
      const Item32 it = decode32(item, a);
      const int nkb = (min(kT, L - it.k * kT) + kKB - 1) / kKB;
      const int set = jl & 1;
      if (jl >= 2) ptx::mbar_wait(&acc_free[set], ((jl >> 1) - 1) & 1, a.err, 181);
      ptx::tc_fence_after();
      for (int kb = 0; kb < nkb; ++kb, ++u) {
        const int sl = u % nst;
        ptx::mbar_wait(&ready[sl], (u / nst) & 1, a.err, 182);
        ptx::tc_fence_after();
        if (leader) {
          const uint32_t s0 = ptx::smem_u32(stage_ptr(u));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = ptx::smem_desc(s0 + kk * 32, 16, 1024, ptx::kSw128);
            const uint64_t bd = ptx::smem_desc(s0 + 4 * kBox + kk * 32, 16, 1024, ptx::kSw128);
            ptx::mma_ss<true>(tmem + set * HP, ad, bd, idesc, (kb | kk) ? 1u : 0u);
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
    const int quad = warp & 3, half = warp >> 2;  // TMEM lane quadrant, column half
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const int r = tid & 31, cc = tid >> 5;  // a box's row (token) and 16-byte piece
    auto warp_arrive = [&](uint64_t *bar) {
      __syncwarp();
      if ((tid & 31) == 0) ptx::mbar_arrive(bar);
    };
    // dt of thread = token tid and A for the H heads of an item, one item
    // ahead
    struct ItemIn {
      float Aq[kMaxH], dtj[kMaxH];
    };
    auto fetch_item = [&](int item) {
      ItemIn in;
#pragma unroll
      for (int q = 0; q < kMaxH; ++q) in.Aq[q] = in.dtj[q] = 0.f;
      if (item >= a.n_items) return in;
      const Item32 it = decode32(item, a);
      const int tok0 = it.k * kT, valid = min(kT, L - tok0);
#pragma unroll
      for (int q = 0; q < kMaxH; ++q) {
        const int h = it.hbase + q;
        if (q < H && SSD_IN_BOUNDS(h < nh && it.b < a.nb, a.err, 180)) {
          in.Aq[q] = a.A[h];
          if (tid < valid) in.dtj[q] = a.dt[((int64_t)it.b * L + tok0 + tid) * nh + h];
        }
      }
      return in;
    };

    // the epilogue of item jl: D[s][(q, p)] -> dstates[b, h, k][p][st 128 + s]
    // (warp: its lane quadrant; T = the item's H P columns split in halves)
    auto epilogue = [&](const Item32 &it, int jl) {
      const int set = jl & 1;
      ptx::mbar_wait(&acc_full[set], (jl >> 1) & 1, a.err, 183);
      ptx::tc_fence_after();
      const int s = it.st * 128 + quad * 32 + (tid & 31);
      const int ncol = HP / 2, c_lo = half * ncol;
      // rows of the slice past S (S = 64: the upper half, whose B boxes were
      // zero-filled) hold nothing to store; whole warps skip them
      for (int c0 = c_lo; c0 < c_lo + ncol && it.st * 128 + quad * 32 < S; c0 += 16) {
        float v[16];
        ptx::tmem_ld16_sync(tmem + lane_base + set * HP + c0, v);
        const int q = c0 / kP, p0 = c0 % kP;
        const int64_t base = ((((int64_t)it.b * nh + it.hbase + q) * nc + it.k) * kP + p0) * S + s;
        if (SSD_IN_BOUNDS(base + 15 * (int64_t)S < (int64_t)a.nb * nh * nc * kP * S, a.err, 181)) {
#pragma unroll
          for (int e = 0; e < 16; ++e) a.dstates[base + (int64_t)e * S] = v[e];
        }
      }
      ptx::tc_fence_before();
      warp_arrive(&acc_free[set]);
    };

    ItemIn in_next = fetch_item(blockIdx.x);
    Item32 prev{0, 0, 0, 0};
    int u = 0, jl = 0;
    for (int item = blockIdx.x; item < a.n_items; item += gridDim.x, ++jl) {
      const Item32 it = decode32(item, a);
      const int tok0 = it.k * kT, valid = min(kT, L - tok0);
      const int nkb = (valid + kKB - 1) / kKB;
      const ItemIn in = in_next;
      in_next = fetch_item(item + gridDim.x);  // in flight while this item runs
      float(*w)[256] = ws[jl & 1];
      float(*wt)[kRowWarps] = warp_tot[jl & 1];
      // the in-chunk cumsums of the item's heads (thread = token; a padding
      // token adds zero, so the chunk total is G at its last real token) and
      // the jump weights.  The stage barriers of the previous item keep every
      // thread past its last use of this parity's arrays (item jl - 2) before
      // they are overwritten.
      float incl[kMaxH];
#pragma unroll
      for (int q = 0; q < kMaxH; ++q) {
        incl[q] = in.Aq[q] * kLog2e * in.dtj[q];
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
          const float t2 = wt[q][w2];
          tot += t2;
          if (w2 < warp) base += t2;
        }
        const float Gj = base + incl[q];
        if (tid < kT) {
          w[q][tid] = tid < valid ? exp2f(tot - Gj) * in.dtj[q] : 0.f;
          const int64_t g0 = (((int64_t)it.b * nh + it.hbase + q) * nc + it.k) * kT;
          if (it.st == 0 && SSD_IN_BOUNDS(g0 + kT <= (int64_t)a.nb * nh * nc * kT, a.err, 185))
            a.G[g0 + tid] = Gj;
        }
      }
      ptx::named_bar_sync(1, kRowThreads);

      for (int kb = 0; kb < nkb; ++kb, ++u) {
        const int sl = u % nst;
        ptx::mbar_wait(&full[sl], (u / nst) & 1, a.err, 184);
        uint8_t *st = stage_ptr(u);
        // read: this thread's 16-byte piece of row r of every box
        float4 v[4 + 2 * kMaxH];
#pragma unroll
        for (int i = 0; i < 4 + 2 * kMaxH; ++i)
          if (i < 4 + 2 * H)
            v[i] = *reinterpret_cast<const float4 *>(st + i * kBox + sw128(r, cc * 16));
        // every thread has read before any writes (in place)
        ptx::named_bar_sync(1, kRowThreads);
        // write: element (row r, columns 4 cc .. 4 cc + 3) of a box to
        // (rows 4 cc .. 4 cc + 3, column r), rounded; x scaled by w of token r
#pragma unroll
        for (int i = 0; i < 4 + 2 * kMaxH; ++i) {
          if (i >= 4 + 2 * H) break;
          const float sc = i < 4 ? 1.f : w[(i - 4) >> 1][kb * kKB + r];
          const float e4[4] = {v[i].x * sc, v[i].y * sc, v[i].z * sc, v[i].w * sc};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            *reinterpret_cast<uint32_t *>(st + i * kBox + sw128(4 * cc + e, r * 4)) =
                to_tf32(e4[e]);
        }
        ptx::fence_async_smem();
        warp_arrive(&ready[sl]);
      }
      if (jl > 0) epilogue(prev, jl - 1);
      prev = it;
    }
    if (jl > 0) epilogue(prev, jl - 1);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, 2 * HP <= 256 ? 256 : 512);
}

// Heads per item: four when the group allows (B is loaded once per four
// heads; 95 us against 127 with two on the fp32 sweep b2 h32 S128 L16384
// T256), else two or
// one.
int cs32_heads(const Dims &d) { return d.hpg % 4 == 0 ? 4 : d.hpg % 2 == 0 ? 2 : 1; }

int cs32_stages(const Dims &d) {
  const int stage_bytes = 4 * kBox + cs32_heads(d) * 2 * kBox;
  return std::min(kMaxSt, (219 * 1024) / stage_bytes);
}

}  // namespace

bool fwd_chunk_state_tf32_supported(const Dims &d) {
  return d.P == kP && d.S % 64 == 0 && (d.T == 128 || d.T == 256) && cs32_stages(d) >= 2;
}

cudaError_t launch_fwd_chunk_state_tf32(const Dims &d, const float *x, const float *B,
                                        const float *dt, const float *A, float *G,
                                        float *dstates, int *err, cudaStream_t st) {
  if (!fwd_chunk_state_tf32_supported(d)) return cudaErrorInvalidValue;
  CUtensorMap tB, tx;
  if (!make_tmap_bl(&tB, B, false, d.b, d.L, d.ng, d.S, kKB) ||
      !make_tmap_bl(&tx, x, false, d.b, d.L, d.nh, d.P, kKB))
    return cudaErrorInvalidValue;
  const int H = cs32_heads(d), nst = cs32_stages(d);
  const int smem = nst * (4 * kBox + H * 2 * kBox) + 1024;
  auto kernel = d.T == 256 ? fwd_chunk_state_tf32<256> : fwd_chunk_state_tf32<128>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  CsArgs32 a;
  a.dt = dt;
  a.A = A;
  a.G = G;
  a.dstates = dstates;
  a.err = err;
  a.L = (int)d.L;
  a.nh = (int)d.nh;
  a.S = (int)d.S;
  a.hpg = (int)d.hpg;
  a.T = (int)d.T;
  a.nc = (int)d.nc;
  a.nb = (int)d.b;
  a.H = H;
  a.n_st = (int)((d.S + 127) / 128);
  a.n_hg = (int)(d.nh / H);
  a.nst = nst;
  const int64_t n_items = d.b * d.nc * a.n_st * a.n_hg;
  if (n_items > 0x7fffffffLL) return cudaErrorInvalidValue;
  a.n_items = (int)n_items;
  const int grid = (int)std::min<int64_t>(n_items, sm_count());
  kernel<<<grid, kThreads, smem, st>>>(tB, tx, a);
  return cudaGetLastError();
}

}  // namespace ssd
