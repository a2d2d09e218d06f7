// Step 2: the jump term of the chunk state update
//
//   dstates[b,h,k][p][s] = sum_{j in chunk k} w_j x[b,j,h,p] B[b,j,g,s],
//   w_j = exp2(G_last,k - G_j) dt_j
//
// ("Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA
// CUDA Tile", section "Mamba-2 architecture", the log-space jump formula
// h_{t+T} = exp(G_last) h_t + (exp(G_last - G) B)^T X, second term.)
//
// Tensor-core kernel (tcgen05).  One CTA per (chunk, 128-wide slice of S,
// head, batch) computes D[s][p] = sum_j B[j][s] (w_j x[j][p]) as an
// M = 128 (s) x N = P MMA with K = the chunk's tokens:
//   - TMA stages 64-token blocks of B (A operand, s contiguous: MN-major) and
//     x (B operand, p contiguous: MN-major) into 128-byte-swizzled shared
//     memory, two stages deep;
//   - the threads scale each x row by w_j in place (a row of the swizzled
//     tile holds one token, so the swizzle does not matter);
//   - one thread issues the MMAs, accumulating in tensor memory (TMEM);
//   - the epilogue reads TMEM lane s and writes dstates[p][s], coalesced
//     along s.
// With fp32 I/O the MMAs run as kind::tf32, which takes K-major operands
// only; there the threads stage both operands transposed (tokens along the
// 128-byte rows), 32 tokens per stage, rounding to tf32.
#include "tc_common.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 128;
constexpr int kKB = 64;   // tokens per pipeline stage
constexpr int kMT = 128;  // s per CTA (MMA M)

template <typename IO>
__global__ void __launch_bounds__(kThreads)
chunk_state_tc(const __grid_constant__ CUtensorMap tm_B, const __grid_constant__ CUtensorMap tm_x,
               const IO *__restrict__ dt, const float *__restrict__ G,
               float *__restrict__ dstates, int *__restrict__ err, int L, int nh, int P, int S,
               int hpg, int T, int nc, int nb) {
  using Tr = IoT<IO>;
  constexpr int kAE = Tr::kAE;
  constexpr int nMb = kMT / kAE;  // A-operand 128-byte blocks along s
  constexpr int kBlk = kKB * 128; // bytes of one 64-row block
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full[2], mmad[2];
  __shared__ uint32_t tmem_slot;
  __shared__ float w[256];

  const int nPb = (P + kAE - 1) / kAE;
  const int stage_bytes = (nMb + nPb) * kBlk;
  const int k = blockIdx.x;
  const int n_st = (S + kMT - 1) / kMT;
  const int h = blockIdx.y / n_st, st_idx = blockIdx.y % n_st;
  const int b = blockIdx.z, g = h / hpg;
  const int s0 = st_idx * kMT;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int tok0 = k * T;
  const int valid = min(T, L - tok0);
  const int nkb = (valid + kKB - 1) / kKB;
  const uint32_t ncols = P <= 32 ? 32 : (P <= 64 ? 64 : 128);

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&mmad[i], 1);
    }
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tm_B);
    ptx::prefetch_tmap(&tm_x);
  }
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_slot, ncols);
    ptx::tmem_relinquish();
  }
  // w_j = exp2(G_last - G_j) dt_j, zero past the end of the sequence.
  const int64_t nG = (int64_t)nb * nh * nc * T, ndt = (int64_t)nb * L * nh;
  const int64_t g0 = ((int64_t)(b * nh + h) * nc + k) * T;
  const float *Gc = G + g0;
  const float Glast = SSD_IN_BOUNDS(g0 + T <= nG, err, 81) ? Gc[T - 1] : 0.f;
  for (int j = tid; j < T; j += kThreads) {
    float v = 0.f;
    const int64_t idt = ((int64_t)b * L + tok0 + j) * nh + h;
    if (j < valid && SSD_IN_BOUNDS(g0 + j < nG && idt < ndt, err, 82))
      v = exp2f(Glast - Gc[j]) * ld_io(dt + idt);
    w[j] = v;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;

  auto issue_loads = [&](int kb) {
    const int s = kb & 1;
    uint8_t *A = smem + s * stage_bytes;
    uint8_t *X = A + nMb * kBlk;
    ptx::mbar_arrive_expect_tx(&full[s], stage_bytes);
    for (int mb = 0; mb < nMb; ++mb)
      ptx::tma_load_4d(A + mb * kBlk, &tm_B, s0 + mb * kAE, g, tok0 + kb * kKB, b, &full[s]);
    for (int pb = 0; pb < nPb; ++pb)
      ptx::tma_load_4d(X + pb * kBlk, &tm_x, pb * kAE, h, tok0 + kb * kKB, b, &full[s]);
  };

  if (tid == 0)
    for (int kb = 0; kb < min(nkb, 2); ++kb) issue_loads(kb);

  const uint32_t idesc = mma_idesc<IO>(128, P, true, true);
  for (int kb = 0; kb < nkb; ++kb) {
    const int s = kb & 1;
    const uint32_t ph = (kb >> 1) & 1;
    uint8_t *A = smem + s * stage_bytes;
    uint8_t *X = A + nMb * kBlk;
    ptx::mbar_wait(&full[s], ph, err, 21);
    // scale the x rows of this block by w_j (16-byte chunks, row = token)
    for (int c = tid; c < nPb * kKB * 8; c += kThreads) {
      const int row = (c >> 3) & (kKB - 1);
      const float ws = w[kb * kKB + row];
      uint4 *p4 = reinterpret_cast<uint4 *>(X + c * 16);
      float v[8];
      unpack16(*p4, v, (IO *)nullptr);
#pragma unroll
      for (int i = 0; i < 16 / Tr::kE; ++i) v[i] *= ws;
      *p4 = pack_op16(v, (IO *)nullptr);
    }
    ptx::fence_async_smem();
    __syncthreads();
    if (tid == 0) {
      ptx::tc_fence_after();
      const uint32_t a0 = ptx::smem_u32(A), x0 = ptx::smem_u32(X);
#pragma unroll
      for (int kk = 0; kk < kKB / Tr::kKmma; ++kk) {
        const uint64_t ad = ptx::smem_desc(a0 + kk * Tr::kKmma * 128, kBlk, 1024, ptx::kSw128);
        const uint64_t bd = ptx::smem_desc(x0 + kk * Tr::kKmma * 128, kBlk, 1024, ptx::kSw128);
        ptx::mma_ss<Tr::kTf32>(tmem, ad, bd, idesc, (kb | kk) ? 1u : 0u);
      }
      ptx::mma_commit(&mmad[s]);
      if (kb + 2 < nkb) {
        ptx::mbar_wait(&mmad[s], ph, err, 22);
        issue_loads(kb + 2);
      }
    }
  }
  // all MMAs done (the last commit tracks every earlier MMA of the thread)
  ptx::mbar_wait(&mmad[(nkb - 1) & 1], ((nkb - 1) >> 1) & 1, err, 23);
  ptx::tc_fence_after();

  const int srow = s0 + warp * 32 + lane;
  const int64_t o0 = ((int64_t)(b * nh + h) * nc + k) * P * S;
  float *out = dstates + o0;
  for (int c0 = 0; c0 < P; c0 += 16) {
    float v[16];
    ptx::tmem_ld16_sync(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
    if (srow < S &&
        SSD_IN_BOUNDS(o0 + (int64_t)(c0 + 15) * S + srow < (int64_t)nb * nh * nc * P * S, err, 83)) {
#pragma unroll
      for (int j = 0; j < 16; ++j) out[(int64_t)(c0 + j) * S + srow] = v[j];
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tmem, ncols);
}

// fp32 I/O: K-major staging by the threads (kind::tf32 has no MN-major mode).
constexpr int kKB32 = 32;  // tokens per stage: one 128-byte row of fp32

__global__ void __launch_bounds__(kThreads)
chunk_state_tf32(const float *__restrict__ x, const float *__restrict__ Bm,
                 const float *__restrict__ dt, const float *__restrict__ G,
                 float *__restrict__ dstates, int *__restrict__ err, int L, int nh, int P, int S,
                 int hpg, int T, int nc, int nb) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t mmad[2];
  __shared__ uint32_t tmem_slot;
  __shared__ float w[256];

  const int aBytes = kMT * 128;                       // A: 128 rows s
  const int stage_bytes = aBytes + ((P * 128 + 1023) & ~1023);  // + X: P rows p
  const int k = blockIdx.x;
  const int n_st = (S + kMT - 1) / kMT;
  const int h = blockIdx.y / n_st, st_idx = blockIdx.y % n_st;
  const int b = blockIdx.z, g = h / hpg;
  const int s0 = st_idx * kMT;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int tok0 = k * T;
  const int valid = min(T, L - tok0);
  const int nkb = (valid + kKB32 - 1) / kKB32;
  const uint32_t ncols = P <= 32 ? 32 : (P <= 64 ? 64 : 128);

  if (tid == 0) {
    ptx::mbar_init(&mmad[0], 1);
    ptx::mbar_init(&mmad[1], 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_slot, ncols);
    ptx::tmem_relinquish();
  }
  const int64_t nG = (int64_t)nb * nh * nc * T, ndt = (int64_t)nb * L * nh;
  const int64_t g0 = ((int64_t)(b * nh + h) * nc + k) * T;
  const float *Gc = G + g0;
  const float Glast = SSD_IN_BOUNDS(g0 + T <= nG, err, 84) ? Gc[T - 1] : 0.f;
  for (int j = tid; j < T; j += kThreads) {
    const int64_t idt = ((int64_t)b * L + tok0 + j) * nh + h;
    w[j] = j < valid && SSD_IN_BOUNDS(g0 + j < nG && idt < ndt, err, 85)
               ? exp2f(Glast - Gc[j]) * dt[idt]
               : 0.f;
  }
  const int64_t nB = (int64_t)nb * L * (nh / hpg) * S, nx = (int64_t)nb * L * nh * P;
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t idesc = ptx::idesc_tf32(128, P, false, false);

  for (int kb = 0; kb < nkb; ++kb) {
    const int s = kb & 1;
    if (kb >= 2) ptx::mbar_wait(&mmad[s], ((kb >> 1) - 1) & 1, err, 24);
    uint8_t *A = smem + s * stage_bytes;
    uint8_t *X = A + aBytes;
    // A[s][j] = B[token j][s] and X[p][j] = w_j x[token j][p], transposed
    // through registers: lane = token j of the block, each lane loads 16
    // bytes (four consecutive s or p) and writes them down four rows at its
    // column, so a warp writes 32 consecutive words of a row (no bank
    // conflicts); every load of the block is issued before the first store.
    constexpr int kAq = (kMT / 4) * kKB32 / kThreads;  // B quads per thread (8)
    constexpr int kXqMax = (128 / 4) * kKB32 / kThreads;  // x quads per thread, P <= 128
    const int nXq = (P / 4) * kKB32;
    float4 bq[kAq], xq[kXqMax];
#pragma unroll
    for (int r = 0; r < kAq; ++r) {
      const int idx = tid + r * kThreads, j = idx % kKB32, q = idx / kKB32;
      const int jt = kb * kKB32 + j;
      const int64_t iB = (((int64_t)b * L + tok0 + jt) * (nh / hpg) + g) * S + s0 + 4 * q;
      bq[r] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (s0 + 4 * q < S && jt < valid && SSD_IN_BOUNDS(iB + 4 <= nB, err, 86))
        bq[r] = *reinterpret_cast<const float4 *>(Bm + iB);
    }
#pragma unroll
    for (int r = 0; r < kXqMax; ++r) {
      const int idx = tid + r * kThreads, j = idx % kKB32, q = idx / kKB32;
      const int jt = kb * kKB32 + j;
      const int64_t ix = (((int64_t)b * L + tok0 + jt) * nh + h) * P + 4 * q;
      xq[r] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (idx < nXq && jt < valid && SSD_IN_BOUNDS(ix + 4 <= nx, err, 87))
        xq[r] = *reinterpret_cast<const float4 *>(x + ix);
    }
#pragma unroll
    for (int r = 0; r < kAq; ++r) {
      const int idx = tid + r * kThreads, j = idx % kKB32, q = idx / kKB32;
      *reinterpret_cast<uint32_t *>(A + sw128(4 * q + 0, j * 4)) = to_tf32(bq[r].x);
      *reinterpret_cast<uint32_t *>(A + sw128(4 * q + 1, j * 4)) = to_tf32(bq[r].y);
      *reinterpret_cast<uint32_t *>(A + sw128(4 * q + 2, j * 4)) = to_tf32(bq[r].z);
      *reinterpret_cast<uint32_t *>(A + sw128(4 * q + 3, j * 4)) = to_tf32(bq[r].w);
    }
#pragma unroll
    for (int r = 0; r < kXqMax; ++r) {
      const int idx = tid + r * kThreads, j = idx % kKB32, q = idx / kKB32;
      if (idx >= nXq) break;
      const float wj = w[kb * kKB32 + j];
      *reinterpret_cast<uint32_t *>(X + sw128(4 * q + 0, j * 4)) = to_tf32(wj * xq[r].x);
      *reinterpret_cast<uint32_t *>(X + sw128(4 * q + 1, j * 4)) = to_tf32(wj * xq[r].y);
      *reinterpret_cast<uint32_t *>(X + sw128(4 * q + 2, j * 4)) = to_tf32(wj * xq[r].z);
      *reinterpret_cast<uint32_t *>(X + sw128(4 * q + 3, j * 4)) = to_tf32(wj * xq[r].w);
    }
    ptx::fence_async_smem();
    __syncthreads();
    if (tid == 0) {
      ptx::tc_fence_after();
      const uint32_t a0 = ptx::smem_u32(A), x0 = ptx::smem_u32(X);
#pragma unroll
      for (int kk = 0; kk < kKB32 / 8; ++kk) {
        const uint64_t ad = ptx::smem_desc(a0 + kk * 32, 16, 1024, ptx::kSw128);
        const uint64_t bd = ptx::smem_desc(x0 + kk * 32, 16, 1024, ptx::kSw128);
        ptx::mma_ss<true>(tmem, ad, bd, idesc, (kb | kk) ? 1u : 0u);
      }
      ptx::mma_commit(&mmad[s]);
    }
  }
  ptx::mbar_wait(&mmad[(nkb - 1) & 1], ((nkb - 1) >> 1) & 1, err, 25);
  ptx::tc_fence_after();

  const int srow = s0 + warp * 32 + lane;
  const int64_t o0 = ((int64_t)(b * nh + h) * nc + k) * P * S;
  float *out = dstates + o0;
  for (int c0 = 0; c0 < P; c0 += 16) {
    float v[16];
    ptx::tmem_ld16_sync(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
    if (srow < S &&
        SSD_IN_BOUNDS(o0 + (int64_t)(c0 + 15) * S + srow < (int64_t)nb * nh * nc * P * S, err, 88)) {
#pragma unroll
      for (int j = 0; j < 16; ++j) out[(int64_t)(c0 + j) * S + srow] = v[j];
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tmem, ncols);
}

template <typename IO>
cudaError_t launch_t(const Dims &d, const void *x, const void *B, const void *dt,
                     const float *G, float *dstates, int *err, cudaStream_t st) {
  const int n_st = (int)((d.S + kMT - 1) / kMT);
  dim3 grid((unsigned)d.nc, (unsigned)(d.nh * n_st), (unsigned)d.b);
  if constexpr (IoT<IO>::kTf32) {
    const int smem = 2 * (kMT * 128 + (int)((d.P * 128 + 1023) & ~1023)) + 1024;
    cudaError_t e = cudaFuncSetAttribute(chunk_state_tf32,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    chunk_state_tf32<<<grid, kThreads, smem, st>>>(
        static_cast<const float *>(x), static_cast<const float *>(B),
        static_cast<const float *>(dt), G, dstates, err, (int)d.L, (int)d.nh,
        (int)d.P, (int)d.S, (int)d.hpg, (int)d.T, (int)d.nc, (int)d.b);
    return cudaGetLastError();
  } else {
    constexpr bool bf = true;
    CUtensorMap tB, tx;
    if (!make_tmap_bl(&tB, B, bf, d.b, d.L, d.ng, d.S, kKB) ||
        !make_tmap_bl(&tx, x, bf, d.b, d.L, d.nh, d.P, kKB))
      return cudaErrorInvalidValue;
    const int nPb = (int)((d.P + IoT<IO>::kAE - 1) / IoT<IO>::kAE);
    const int smem = 2 * (kMT / IoT<IO>::kAE + nPb) * kKB * 128 + 1024;
    auto kern = chunk_state_tc<IO>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, st>>>(tB, tx, static_cast<const IO *>(dt), G, dstates,
                                       err, (int)d.L, (int)d.nh, (int)d.P,
                                       (int)d.S, (int)d.hpg, (int)d.T, (int)d.nc, (int)d.b);
    return cudaGetLastError();
  }
}

}  // namespace

cudaError_t launch_chunk_state(const Dims &d, ssd_dtype io, const void *x, const void *B,
                               const void *dt, const float *G, float *dstates, int *err,
                               cudaStream_t st) {
  return io == SSD_BF16 ? launch_t<__nv_bfloat16>(d, x, B, dt, G, dstates, err, st)
                        : launch_t<float>(d, x, B, dt, G, dstates, err, st);
}

}  // namespace ssd
