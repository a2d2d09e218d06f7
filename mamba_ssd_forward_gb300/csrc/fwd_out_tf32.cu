// Forward path, output pass with fp32 I/O (kind::tf32 MMAs, fp32
// accumulation): the chunked output equation of "Accelerating Mamba-2 with
// High-Performance Forward Pass Kernels in NVIDIA CUDA Tile", section
// "Mamba-2 architecture" (the compute_out step),
//
//   y_i = exp2(G_i) (h_k c_i) + sum_{j<=i in chunk} (c_i . B_j) exp2(G_i - G_j) dt_j x_j
//         + D x_i,
//
// G the in-chunk cumsum of A dt in log2 units, h_k the chunk's start state.
// As in the bf16 output pass (fwd_out.cu) the decay of the in-chunk sum is
// factored about an anchor alpha = rint(G_last / 2):
// exp2(G_i - G_j) = u_i v'_j with u_i = exp2(G_i - alpha), v'_j =
// exp2(alpha - G_j), so the masked C B^T of the chunk carries no decay and is
// shared unchanged by every head of the group; per head the x rows are only
// scaled by v_j = v'_j dt_j, and with exp2(G_i) = u_i 2^alpha
//
//   y_i = u_i [ c_i . (2^alpha h_k) + sum_{j<=i} (c_i . B_j) v_j x_j ] + D x_i:
//
// one accumulation per head, C (2^alpha h)^T + (C B^T masked) Xh, with the
// start states stored times 2^alpha by the state pass (an exact power of
// two; alpha = 0 when the chunk's total decay exceeds 2^-180).  A chunk whose
// decay is too steep for bounded factors (that, or a real token's factor
// below 2^-120) takes an exact per-element path for the in-chunk sum on the
// CUDA cores instead (rare, slow, exact).
//
// kind::tf32 takes K-major operands only, and every operand is rounded to
// tf32 (nearest) before the tensor core sees it: C as the row warps move it
// into tensor memory, B in shared memory as it lands, the start states by
// the state pass that stores them, x while it is transposed, C B^T in
// tensor memory.
//
// One CTA per (128-row tile t of a chunk, slice of hs heads of one group,
// chunk, batch), 1 CTA per SM, everything staged through one ring of 16 KB
// stages:
//   producer warp: C of the tile (atoms of 32 s, rows = the tile's tokens),
//     B of tokens 0 .. 128 (t + 1) - 1 per atom of S, then per head its x
//     (64 tokens per stage, as landed: p contiguous) and its start state
//     (two atoms of S per stage);
//   MMA warp: C B^T of the tile (A = C from tensor memory) into tensor
//     memory, fp32, columns = tokens; per head into one of two accumulator
//     sets (C B^T masked) Xh (A = C B^T, B = the row warps' transposed x
//     atoms) + C (2^alpha h)^T (A = C);
//   row warps (8): C into tensor memory (rounded), the B stages rounded in
//     place; C B^T masked (j > i -> 0) and rounded in place; per head its
//     factors, the transposition of each 32-token x atom into K-major Xh^T
//     (tokens along the 128-byte rows, scaled by v_j, rounded), and the
//     previous head's epilogue y = u_i Acc_i + D x_i.
// At S > 128, C's first 128 columns of S sit in tensor memory and the rest
// in shared memory (the 512 tensor-memory columns hold C B^T, 128 of C and
// the two accumulator sets); those MMAs read A from shared memory.
// Supported: P = 64, S a multiple of 32 up to 256, T in {128, 256}.
#include "fwd.cuh"

namespace ssd {
namespace {

constexpr int kRowWarps = 8;
constexpr int kRowThreads = kRowWarps * 32;
constexpr int kThreads = kRowThreads + 64;
constexpr int kProducerWarp = kRowWarps, kMmaWarp = kRowWarps + 1;
constexpr int kP = 64;
constexpr int kStage = 16384;     // one ring stage: C or B (128 rows x 32 fp32 of
                                  // S), two state atoms, or 64 tokens of x
constexpr int kHAtom = 64 * 128;  // start state: 64 rows p x 32 fp32 of S
constexpr int kXAtom = 64 * 128;  // x of 32 tokens: two 32 x 32 boxes (p halves)
constexpr int kMaxSlots = 12;
constexpr float kSpanMax = 180.f;
constexpr float kMinFactor = 7.52316384526264e-37f;  // 2^-120

// Tensor-memory columns: C B^T of the tile at [0, 128 (t + 1)); C of the
// tile at [256, 256 + S); accumulator set s at 384 + 64 s.
constexpr uint32_t kColC = 256;
__device__ __forceinline__ uint32_t acc_col(int set) { return 384u + 64u * (uint32_t)set; }

struct OutArgs32 {
  const float *x, *dt, *D;
  const float *G;  // in-chunk cumsums, log2 units, [b, nh, nc * T]
  float *y;
  int *err;
  int L, nh, S, hpg, T, nc, hs, nslot, nb;
};

__device__ __forceinline__ float tf32_rn(float v) { return __uint_as_float(to_tf32(v)); }

// kSplitC: dstate above 128, C split between tensor and shared memory (a
// compile-time choice, so that the MMA warp's issue loop at dstate <= 128
// carries no test of where C lies)
template <int kT, bool kSplitC>
__global__ void __launch_bounds__(kThreads, 1)
fwd_out_tf32(const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_B,
             const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_st,
             const __grid_constant__ CUtensorMap tm_y, const OutArgs32 a) {
  constexpr int nT = kT / 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  // full: a state stage landed (MMA waits); xfull: a C, B or x stage landed
  // (row warps wait); scaled: the row warps rounded a B stage or transposed
  // an x stage in place; empty: the MMAs reading a B, x or state stage are
  // done; xrel: every row warp is done with a C stage; c_ready: C is in
  // tensor memory
  __shared__ __align__(8) uint64_t c_ready, c2_full, full[kMaxSlots], xfull[kMaxSlots],
      scaled[kMaxSlots], empty[kMaxSlots], xrel[kMaxSlots], sc_done, pack_done, acc_full[2],
      acc_free[2];
  __shared__ uint32_t tmem_slot;
  // per head (by head parity): G and dt of every token, v_j, alpha, path
  __shared__ __align__(16) float Gs[2][256];
  __shared__ __align__(16) float dts[2][256];
  __shared__ __align__(16) float vs[2][256];
  __shared__ float alphas[2];
  __shared__ int steeps[2];
  __shared__ int warp_ok[kRowWarps];

  const int L = a.L, nh = a.nh, S = a.S, hs = a.hs, nslot = a.nslot;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int t = blockIdx.x % nT;             // row tile of the chunk
  const int hbase = (blockIdx.x / nT) * hs;  // first head of the slice
  const int k = blockIdx.y, b = blockIdx.z;
  const int g = hbase / a.hpg;
  const int tok0 = k * kT;
  const int valid = min(kT, L - tok0);
  if (t * 128 >= valid) return;  // the whole tile lies past the sequence (uniform)
  const int nS = S / 32;             // K atoms of S
  const int nCt = kSplitC ? 4 : nS;  // atoms of C in tensor memory (S < 128 of it)
  const int nCs = kSplitC ? nS - 4 : 0;  // atoms of C resident in shared memory (S > 128)
  const int nHs = (nS + 1) / 2;      // state stages per head
  const int nJ = 4 * (t + 1);        // 32-token atoms of the in-chunk sum
  const int nXs = nJ / 2;            // x stages per head (64 tokens each)
  uint8_t *Cres = smem;  // C atoms 4 .. nS - 1 of the tile (S > 128), 16 KB each
  uint8_t *ring = smem + nCs * kStage;
  uint8_t *ystage = ring + nslot * kStage;  // y of one head: two 16 KB boxes
  auto slot_ptr = [&](int u) { return ring + (u % nslot) * kStage; };

  if (tid == 0) {
    ptx::mbar_init(&c_ready, kRowWarps);
    ptx::mbar_init(&c2_full, 1);
    for (int i = 0; i < nslot; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&xfull[i], 1);
      ptx::mbar_init(&scaled[i], kRowWarps);
      ptx::mbar_init(&empty[i], 1);
      ptx::mbar_init(&xrel[i], kRowWarps);
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
    ptx::tmem_alloc(&tmem_slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const bool leader = (tid & 31) == 0;
  const int n_pa = nS * (t + 1);  // B stages

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (leader) {
      ptx::prefetch_tmap(&tm_C);
      ptx::prefetch_tmap(&tm_B);
      ptx::prefetch_tmap(&tm_x);
      ptx::prefetch_tmap(&tm_st);
      ptx::prefetch_tmap(&tm_y);
    }
    __syncwarp();
    int u = 0;
    // the previous use of a slot was released on empty (its reader the MMA
    // warp) or on xrel (the row warps): one bit per slot says which, one
    // parity bit per slot and barrier says which phase to wait for
    uint32_t prev_x = 0, epar = 0, rpar = 0;
    auto acquire = [&](int code, bool x_stage) {
      const int sl = u % nslot;
      if (u >= nslot) {
        if ((prev_x >> sl) & 1) {
          ptx::mbar_wait(&xrel[sl], (rpar >> sl) & 1, a.err, code);
          rpar ^= 1u << sl;
        } else {
          ptx::mbar_wait(&empty[sl], (epar >> sl) & 1, a.err, code);
          epar ^= 1u << sl;
        }
      }
      prev_x = x_stage ? (prev_x | (1u << sl)) : (prev_x & ~(1u << sl));
    };
    for (int sb = 0; sb < nCt; ++sb, ++u) {
      acquire(159, true);
      if (leader) {
        ptx::mbar_arrive_expect_tx(&xfull[u % nslot], kStage);
        ptx::tma_load_4d(slot_ptr(u), &tm_C, sb * 32, g, tok0 + t * 128, b, &xfull[u % nslot]);
      }
      __syncwarp();
    }
    if (kSplitC && leader) {
      ptx::mbar_arrive_expect_tx(&c2_full, nCs * kStage);
      for (int i = 0; i < nCs; ++i)
        ptx::tma_load_4d(Cres + i * kStage, &tm_C, (nCt + i) * 32, g, tok0 + t * 128, b, &c2_full);
    }
    __syncwarp();
    for (int sb = 0; sb < nS; ++sb)
      for (int th = 0; th <= t; ++th, ++u) {
        acquire(160, false);
        if (leader) {
          ptx::mbar_arrive_expect_tx(&xfull[u % nslot], kStage);
          ptx::tma_load_4d(slot_ptr(u), &tm_B, sb * 32, g, tok0 + th * 128, b, &xfull[u % nslot]);
        }
        __syncwarp();
      }
    for (int q = 0; q < hs; ++q) {
      const int h = hbase + q;
      const int row = (b * nh + h) * a.nc + k;  // this head's start state
      for (int xs = 0; xs < nXs; ++xs, ++u) {
        acquire(162, false);
        if (leader) {
          // four boxes of 32 tokens x 32 p: token half ai, p half ph at
          // ai * 8 KB + ph * 4 KB
          ptx::mbar_arrive_expect_tx(&xfull[u % nslot], kStage);
          for (int ai = 0; ai < 2; ++ai)
            for (int ph = 0; ph < 2; ++ph)
              ptx::tma_load_4d(slot_ptr(u) + ai * kXAtom + ph * 4096, &tm_x, ph * 32, h,
                               tok0 + xs * 64 + ai * 32, b, &xfull[u % nslot]);
        }
        __syncwarp();
      }
      for (int hh = 0; hh < nHs; ++hh, ++u) {
        acquire(161, false);
        if (leader) {
          // the start states come from the preceding kernel (the state
          // pass), which may still be running when this CTA starts
          if (q == 0 && hh == 0) ptx::griddep_wait();
          const int na = min(2, nS - 2 * hh);
          ptx::mbar_arrive_expect_tx(&full[u % nslot], na * kHAtom);
          for (int ai = 0; ai < na; ++ai)
            ptx::tma_load_3d(slot_ptr(u) + ai * kHAtom, &tm_st, (2 * hh + ai) * 32, 0, row,
                             &full[u % nslot]);
        }
        __syncwarp();
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    uint32_t fpar = 0, spar = 0;  // parity of the next wait, one bit per slot
    ptx::mbar_wait(&c_ready, 0, a.err, 163);
    ptx::tc_fence_after();
    int u = nCt;  // the C stages went to the row warps
    const uint32_t idCB = ptx::idesc_tf32(128, 128, false, false);
    for (int sb = 0; sb < nS; ++sb)
      for (int th = 0; th <= t; ++th, ++u) {
        const int sl = u % nslot;
        ptx::mbar_wait(&scaled[sl], (spar >> sl) & 1, a.err, 164);
        spar ^= 1u << sl;
        ptx::tc_fence_after();
        if (leader) {
          const uint32_t b0 = ptx::smem_u32(slot_ptr(u));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = ptx::smem_desc(b0 + kk * 32, 16, 1024, ptx::kSw128);
            if (!kSplitC || sb < nCt) {
              ptx::mma_ts_tf32(tmem + 128 * th, tmem + kColC + sb * 32 + kk * 8, bd, idCB,
                               (sb | kk) ? 1u : 0u);
            } else {
              const uint64_t cd = ptx::smem_desc(ptx::smem_u32(Cres + (sb - nCt) * kStage) +
                                                     kk * 32,
                                                 16, 1024, ptx::kSw128);
              ptx::mma_ss<true>(tmem + 128 * th, cd, bd, idCB, 1u);
            }
          }
          ptx::mma_commit(&empty[sl]);
        }
        __syncwarp();
      }
    if (leader) ptx::mma_commit(&sc_done);
    __syncwarp();
    const uint32_t idY = ptx::idesc_tf32(128, kP, false, false);
    ptx::mbar_wait(&pack_done, 0, a.err, 165);
    for (int q = 0; q < hs; ++q) {
      const int set = q & 1;
      if (q >= 2) ptx::mbar_wait(&acc_free[set], ((q >> 1) - 1) & 1, a.err, 166);
      ptx::tc_fence_after();
      // Acc = (C B^T masked) Xh over the x stages first (transposed in place
      // by the row warps; no MMA for a steep head, whose epilogue forms the
      // in-chunk sum itself)
      bool steep = false;
      for (int xs = 0; xs < nXs; ++xs, ++u) {
        const int sl = u % nslot;
        ptx::mbar_wait(&scaled[sl], (spar >> sl) & 1, a.err, 168);
        spar ^= 1u << sl;
        ptx::tc_fence_after();
        steep = steeps[q & 1] != 0;
        if (leader) {
          if (!steep) {
            const uint32_t x0 = ptx::smem_u32(slot_ptr(u));
            for (int ai = 0; ai < 2; ++ai)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t xd =
                    ptx::smem_desc(x0 + ai * kXAtom + kk * 32, 16, 1024, ptx::kSw128);
                ptx::mma_ts_tf32(tmem + acc_col(set), tmem + (2 * xs + ai) * 32 + kk * 8, xd,
                                 idY, (xs | ai | kk) ? 1u : 0u);
              }
          }
          ptx::mma_commit(&empty[sl]);
        }
        __syncwarp();
      }
      // Acc += C (2^alpha h)^T over the state stages (the first MMA of a
      // steep head starts the accumulator)
      for (int hh = 0; hh < nHs; ++hh, ++u) {
        const int sl = u % nslot;
        ptx::mbar_wait(&full[sl], (fpar >> sl) & 1, a.err, 167);
        fpar ^= 1u << sl;
        ptx::tc_fence_after();
        if (leader) {
          const uint32_t h0 = ptx::smem_u32(slot_ptr(u));
          const int na = min(2, nS - 2 * hh);
          for (int ai = 0; ai < na; ++ai) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t hd =
                  ptx::smem_desc(h0 + ai * kHAtom + kk * 32, 16, 1024, ptx::kSw128);
              const int sa = 2 * hh + ai;  // atom of S
              const uint32_t accf = (steep && (hh | ai | kk) == 0) ? 0u : 1u;
              if (!kSplitC || sa < nCt) {
                ptx::mma_ts_tf32(tmem + acc_col(set), tmem + kColC + sa * 32 + kk * 8, hd, idY,
                                 accf);
              } else {
                const uint64_t cd = ptx::smem_desc(ptx::smem_u32(Cres + (sa - nCt) * kStage) +
                                                       kk * 32,
                                                   16, 1024, ptx::kSw128);
                ptx::mma_ss<true>(tmem + acc_col(set), cd, hd, idY, accf);
              }
            }
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
    const int lrow = quad * 32 + (tid & 31);  // row of the tile = TMEM lane
    const int i_rel = t * 128 + lrow;          // chunk-relative row
    auto warp_arrive = [&](uint64_t *bar) {
      __syncwarp();
      if ((tid & 31) == 0) ptx::mbar_arrive(bar);
    };
    // round 16 KB of fp32 operand data in place (any layout)
    auto round_block = [&](uint8_t *p, int bytes) {
      for (int o = tid * 16; o < bytes; o += kRowThreads * 16) {
        float4 v = *reinterpret_cast<const float4 *>(p + o);
        v.x = tf32_rn(v.x);
        v.y = tf32_rn(v.y);
        v.z = tf32_rn(v.z);
        v.w = tf32_rn(v.w);
        *reinterpret_cast<float4 *>(p + o) = v;
      }
    };

    // C of the tile into tensor memory, rounded (warp: its lane quadrant, 16
    // of the 32 columns of each atom), then the B stages rounded as they land
    uint32_t xpar = 0;  // parity of the next wait on xfull[slot], one bit per slot
    int u = 0;
    for (int sb = 0; sb < nCt; ++sb, ++u) {
      const int sl = u % nslot;
      ptx::mbar_wait(&xfull[sl], (xpar >> sl) & 1, a.err, 169);
      xpar ^= 1u << sl;
      uint32_t r[16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 v =
            *reinterpret_cast<const uint4 *>(slot_ptr(u) + sw128(lrow, (half * 4 + c) * 16));
        r[4 * c] = to_tf32(__uint_as_float(v.x));
        r[4 * c + 1] = to_tf32(__uint_as_float(v.y));
        r[4 * c + 2] = to_tf32(__uint_as_float(v.z));
        r[4 * c + 3] = to_tf32(__uint_as_float(v.w));
      }
      warp_arrive(&xrel[sl]);  // the values are in registers: the stage may go
      ptx::tmem_stu<16>(tmem + lane_base + kColC + sb * 32 + half * 16, r);
    }
    if (kSplitC) {
      // C's atoms past the first 128 of S stay in shared memory, rounded in
      // place
      ptx::mbar_wait(&c2_full, 0, a.err, 175);
      round_block(Cres, nCs * kStage);
      ptx::fence_async_smem();
    }
    ptx::tmem_st_wait();
    ptx::tc_fence_before();
    warp_arrive(&c_ready);
    for (; u < nCt + n_pa; ++u) {
      const int sl = u % nslot;
      ptx::mbar_wait(&xfull[sl], (xpar >> sl) & 1, a.err, 170);
      xpar ^= 1u << sl;
      round_block(slot_ptr(u), kStage);
      ptx::fence_async_smem();
      warp_arrive(&scaled[sl]);
    }

    // C B^T of the tile: j > i masked to zero, the rest rounded to tf32 in
    // place (warp: its lane quadrant, half the tile's columns)
    ptx::mbar_wait(&sc_done, 0, a.err, 171);
    ptx::tc_fence_after();
    {
      const int ncol = 128 * (t + 1), c_lo = half * (ncol / 2), c_hi = c_lo + ncol / 2;
      for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
        uint32_t r[16];
        ptx::tmem_ld16(tmem + lane_base + c0, r);
        ptx::tmem_ld_wait();
        ptx::reg_fence(r);
#pragma unroll
        for (int e = 0; e < 16; ++e)
          r[e] = (c0 + e <= i_rel) ? to_tf32(__uint_as_float(r[e])) : 0u;
        ptx::tmem_stu<16>(tmem + lane_base + c0, r);
      }
      ptx::tmem_st_wait();
    }
    ptx::tc_fence_before();
    warp_arrive(&pack_done);

    // G and dt come from earlier kernels: wait until the preceding grids are
    // complete
    ptx::griddep_wait();
    // a head's inputs for thread = token j (< T), fetched one head ahead
    struct HeadIn {
      float Gj, dtj, Glast, D;
    };
    auto fetch_head = [&](int q) {
      HeadIn r{0.f, 0.f, 0.f, 0.f};
      const int h = hbase + q;
      const int64_t bhk = ((int64_t)b * nh + h) * a.nc + k;
      if (SSD_IN_BOUNDS(h < nh && bhk < (int64_t)a.nb * nh * a.nc, a.err, 160)) {
        const float *Gc = a.G + bhk * kT;
        if (tid < kT) r.Gj = Gc[tid];
        r.Glast = Gc[kT - 1];
        if (tid < valid) r.dtj = a.dt[((int64_t)b * L + tok0 + tid) * nh + h];
        r.D = a.D ? a.D[h] : 0.f;
      }
      return r;
    };
    // factors and path of head q into the parity-(q & 1) arrays.  The first
    // barrier keeps every write behind the reads of head q - 2's epilogue
    // (same parity), which the slowest row warps may still be doing; the
    // second makes the arrays visible to all.
    auto prep_head = [&](int q, const HeadIn &in) {
      const int pb = q & 1;
      // the anchor the state pass scaled the stored start state by
      const float alpha = -in.Glast <= kSpanMax ? rintf(0.5f * in.Glast) : 0.f;
      const float vj = in.dtj > 0.f ? exp2f(alpha - in.Gj) * in.dtj : 0.f;
      const bool ok = in.dtj == 0.f || vj >= kMinFactor;
      const int all_ok = __all_sync(0xffffffffu, ok);
      ptx::named_bar_sync(1, kRowThreads);
      if ((tid & 31) == 0) warp_ok[warp] = all_ok;
      if (tid < kT) {
        Gs[pb][tid] = in.Gj;
        dts[pb][tid] = in.dtj;
        vs[pb][tid] = vj;
      }
      ptx::named_bar_sync(1, kRowThreads);
      if (tid == 0) {
        // read by the MMA warp after this thread's next arrival on scaled,
        // and by the epilogue of head q, behind head q + 1's barriers
        int okall = 1;
#pragma unroll
        for (int w2 = 0; w2 < kRowWarps; ++w2) okall &= warp_ok[w2];
        steeps[pb] = !(okall && -in.Glast <= kSpanMax);
        alphas[pb] = alpha;
      }
    };

    // the epilogue of head q: y = u_i Acc_i + D x_i for this thread's row
    // and 32 columns (x_i as landed, kept from the transposition of its atom)
    auto epilogue = [&](int q, float Dh, const uint4 (&xk)[8]) {
      const int set = q & 1, pb = q & 1, h = hbase + q;
      float xi[32];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        xi[4 * m] = __uint_as_float(xk[m].x);
        xi[4 * m + 1] = __uint_as_float(xk[m].y);
        xi[4 * m + 2] = __uint_as_float(xk[m].z);
        xi[4 * m + 3] = __uint_as_float(xk[m].w);
      }
      ptx::mbar_wait(&acc_full[set], (q >> 1) & 1, a.err, 172);
      ptx::tc_fence_after();
      const bool steep = steeps[pb] != 0;
      uint32_t ac[32];
      ptx::tmem_ld16(tmem + lane_base + acc_col(set) + 32 * half,
                     *reinterpret_cast<uint32_t(*)[16]>(ac));
      ptx::tmem_ld16(tmem + lane_base + acc_col(set) + 32 * half + 16,
                     *reinterpret_cast<uint32_t(*)[16]>(ac + 16));
      ptx::tmem_ld_wait();
      ptx::reg_fence(ac);
      const float Gi = Gs[pb][min(i_rel, kT - 1)];
      const float ui = exp2f(Gi - alphas[pb]);
      float yv[32];
      if (!steep) {
        ptx::tc_fence_before();
        warp_arrive(&acc_free[set]);  // the accumulators may take head q + 2
#pragma unroll
        for (int c = 0; c < 32; ++c) yv[c] = fmaf(Dh, xi[c], ui * __uint_as_float(ac[c]));
      } else {
        // exact per-element path: the inter-chunk term from the accumulator
        // (C (2^alpha h)^T only), the in-chunk sum from the masked C B^T of
        // this row's lane and the raw x rows (L2), every factor exact
#pragma unroll
        for (int c = 0; c < 32; ++c) yv[c] = fmaf(Dh, xi[c], ui * __uint_as_float(ac[c]));
        const int jmax_warp = t * 128 + quad * 32 + 31;  // the warp's last row
        for (int j0 = 0; j0 <= jmax_warp; j0 += 16) {
          uint32_t cb[16];
          ptx::tmem_ld16(tmem + lane_base + j0, cb);
          ptx::tmem_ld_wait();
          ptx::reg_fence(cb);
          for (int e = 0; e < 16; ++e) {
            const int j = j0 + e;
            if (j >= valid) break;
            const float s = j <= i_rel
                                ? __uint_as_float(cb[e]) * exp2f(Gi - Gs[pb][j]) * dts[pb][j]
                                : 0.f;
            const int64_t xj = (((int64_t)b * L + tok0 + j) * nh + h) * kP + 32 * half;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              const float4 v = *reinterpret_cast<const float4 *>(a.x + xj + 4 * m);
              yv[4 * m] = fmaf(s, v.x, yv[4 * m]);
              yv[4 * m + 1] = fmaf(s, v.y, yv[4 * m + 1]);
              yv[4 * m + 2] = fmaf(s, v.z, yv[4 * m + 2]);
              yv[4 * m + 3] = fmaf(s, v.w, yv[4 * m + 3]);
            }
          }
        }
        ptx::tc_fence_before();
        warp_arrive(&acc_free[set]);
      }
      // y of the tile through the staging buffer (two boxes of 128 rows x
      // 32 p), stored by TMA (rows past the sequence are clipped); the
      // previous head's store must have read the buffer first
      if (tid == 0) ptx::bulk_wait_read<0>();
      ptx::named_bar_sync(2, kRowThreads);
      uint8_t *yt = ystage + half * kStage;
#pragma unroll
      for (int m = 0; m < 8; ++m)
        *reinterpret_cast<float4 *>(yt + sw128(lrow, m * 16)) =
            make_float4(yv[4 * m], yv[4 * m + 1], yv[4 * m + 2], yv[4 * m + 3]);
      ptx::fence_async_smem();
      ptx::named_bar_sync(2, kRowThreads);
      if (tid == 0) {
        for (int ph = 0; ph < 2; ++ph)
          ptx::tma_store_4d(&tm_y, ystage + ph * kStage, ph * 32, h, tok0 + t * 128, b);
        ptx::bulk_commit();
      }
    };

    // Per head q: its factors, the transposition of its x atoms into Xh^T,
    // then the previous head's epilogue (head q's MMAs overlap it).
    const int jl = tid & 31, pc = tid >> 5;  // a box's row (token) and 16-byte piece
    HeadIn in_next = fetch_head(0);
    float D_prev = 0.f;
    uint4 xk[8], xk_prev[8];  // this thread's x row segment (head q, head q - 1)
    for (int q = 0; q < hs; ++q) {
      const HeadIn in = in_next;
      if (q + 1 < hs) in_next = fetch_head(q + 1);
      prep_head(q, in);
      const int pb = q & 1;
      for (int xs = 0; xs < nXs; ++xs, ++u) {
        const int sl = u % nslot;
        ptx::mbar_wait(&xfull[sl], (xpar >> sl) & 1, a.err, 173);
        xpar ^= 1u << sl;
        uint8_t *st = slot_ptr(u);
        // read: this thread's 16-byte piece of row jl of the four boxes, and
        // the warp's own rows for D x_i (raw) when they lie in this stage
        float4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          v[i] = *reinterpret_cast<const float4 *>(st + i * 4096 + sw128(jl, pc * 16));
#pragma unroll
        for (int ai = 0; ai < 2; ++ai)
          if (2 * xs + ai == 4 * t + quad) {
            const uint8_t *xr = st + ai * kXAtom + half * 4096;
#pragma unroll
            for (int m = 0; m < 8; ++m)
              xk[m] = *reinterpret_cast<const uint4 *>(xr + sw128(tid & 31, m * 16));
          }
        // every row thread has read before any writes (in place)
        ptx::named_bar_sync(3, kRowThreads);
        // write: element (token jl, p columns 4 pc .. +3 of box (ai, ph)) to
        // (rows 4 pc .. +3, column jl), scaled by v_j and rounded: each
        // 32-token atom becomes K-major Xh^T, 64 rows of p
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float w = vs[pb][(2 * xs + (i >> 1)) * 32 + jl];
          const float e4[4] = {v[i].x * w, v[i].y * w, v[i].z * w, v[i].w * w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            *reinterpret_cast<uint32_t *>(st + i * 4096 + sw128(4 * pc + e, jl * 4)) =
                to_tf32(e4[e]);
        }
        ptx::fence_async_smem();
        warp_arrive(&scaled[sl]);
      }
      u += nHs;  // the state stages go straight to the MMA warp
      if (q > 0) epilogue(q - 1, D_prev, xk_prev);
      D_prev = in.D;
#pragma unroll
      for (int m = 0; m < 8; ++m) xk_prev[m] = xk[m];
    }
    if (hs > 0) epilogue(hs - 1, D_prev, xk_prev);
    if (tid == 0) ptx::bulk_wait<0>();  // every y store complete
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, 512);
}

struct OutSmem32 {
  int nslot, smem;
};
// The ring and the y staging within 220 KB of dynamic
// shared memory (1 KB of it alignment slack; the static arrays, about 7 KB,
// sit beside it).
OutSmem32 out_smem32(const Dims &d) {
  OutSmem32 m;
  const int c_res = (int)std::max<int64_t>(0, (d.S - 128) / 32) * kStage;
  const int room = (220 * 1024 - 1024 - c_res - 2 * kStage) / kStage;
  m.nslot = std::min(kMaxSlots, room);
  m.smem = c_res + m.nslot * kStage + 2 * kStage + 1024;
  return m;
}

}  // namespace

bool fwd_out_tf32_supported(const Dims &d) {
  if (d.P != kP || d.S % 32 || d.S < 32 || d.S > 256 || (d.T != 128 && d.T != 256))
    return false;
  if (d.nc > 65535 || d.b > 65535) return false;
  // a head's state and x stages in flight, plus one
  return out_smem32(d).nslot >= 4;
}

bool fwd_out_tf32_heads_ok(const Dims &d, int hs) {
  return fwd_out_tf32_supported(d) && hs >= 1 && hs <= d.hpg && d.hpg % hs == 0 &&
         (d.nh / hs) * (d.T / 128) <= 65535;
}

// Heads per CTA: the divisor of the heads per group minimising the busiest
// SM's cost, waves of CTAs times a CTA's cost: its loads (C and B of the tile
// once, per head its state, x and y) plus a fixed start-up of about 8 us (C
// and B of the tile must arrive, C B^T be formed and masked before the first
// head; counted as the 192 KB an SM streams in that time), 10% more when
// there are fewer than three waves of CTAs (the longer second row tile of a
// chunk then balances out less well).  Measured on the fp32 sweep (b2 h32
// S128 L16384 T256): 4 / 8 / 16 / 32 heads per CTA take 329 / 270 / 250 /
// 266 us; the model picks 16.
int fwd_out_tf32_heads(const Dims &d) {
  const int64_t sms = sm_count();
  const int nT = (int)(d.T / 128);
  int best = 1;
  double best_cost = 1e300;
  for (int hs = 1; hs <= d.hpg; ++hs) {
    if (!fwd_out_tf32_heads_ok(d, hs)) continue;
    const int64_t ctas = d.b * d.nc * nT * (d.nh / hs);
    const double per_cta = 192.0 * 1024 + 4.0 * (128.0 * d.S + d.T * d.S) +
                           hs * 4.0 * (d.S * 64.0 + d.T * 64.0 + 128.0 * 64.0);
    const double cost = (double)((ctas + sms - 1) / sms) * per_cta * (ctas < 3 * sms ? 1.1 : 1.0);
    if (cost < best_cost * 0.999) {
      best_cost = cost;
      best = hs;
    }
  }
  return best;
}

cudaError_t launch_fwd_out_tf32(const Dims &d, const float *x, const float *B, const float *C,
                                const float *dt, const float *G, const float *states,
                                const float *D, float *y, int hs, int *err, cudaStream_t st) {
  if (!fwd_out_tf32_heads_ok(d, hs)) return cudaErrorInvalidValue;
  CUtensorMap tC, tB, tx, tS, tY;
  if (!make_tmap_bl(&tC, C, false, d.b, d.L, d.ng, d.S, 128) ||
      !make_tmap_bl(&tB, B, false, d.b, d.L, d.ng, d.S, 128) ||
      !make_tmap_bl(&tx, x, false, d.b, d.L, d.nh, d.P, 32) ||
      !make_tmap_bl(&tY, y, false, d.b, d.L, d.nh, d.P, 128))
    return cudaErrorInvalidValue;
  {
    // start states as [b * nh * nc][P][S] fp32; one box = 64 rows of P x 32 of S
    const uint64_t dims[3] = {(uint64_t)d.S, (uint64_t)d.P, (uint64_t)(d.b * d.nh * d.nc)};
    const uint64_t strides[2] = {(uint64_t)d.S * 4, (uint64_t)(d.S * d.P * 4)};
    const uint32_t box[3] = {32u, 64u, 1u};
    if (!make_tmap_sw128(&tS, states, false, 3, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  const OutSmem32 m = out_smem32(d);
  const bool split = d.S > 128;
  auto kernel = d.T == 256 ? (split ? fwd_out_tf32<256, true> : fwd_out_tf32<256, false>)
                           : (split ? fwd_out_tf32<128, true> : fwd_out_tf32<128, false>);
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, m.smem);
  if (e != cudaSuccess) return e;
  OutArgs32 a;
  a.x = x;
  a.dt = dt;
  a.D = D;
  a.G = G;
  a.y = y;
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
  // programmatic stream serialisation: the producer and the row warps wait
  // on the device before reading the start states and G
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((d.nh / hs) * (d.T / 128)), (unsigned)d.nc, (unsigned)d.b);
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
