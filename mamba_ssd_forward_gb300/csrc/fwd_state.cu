// Forward path, state pass (bf16 I/O): the page's fwd_pass_state ("Kernel 2"
// of "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in
// NVIDIA CUDA Tile"), with the in-chunk cumulative sum ("Kernel 1") fused in.
//
// One CTA per (128-wide slice of S, head, batch) walks the chunks in order:
//   G_j     = log2(e) * sum_{t<=j in chunk} A dt_t          (block scan)
//   states[k] = h                                          (start of chunk)
//   h       = exp2(G_last) h + sum_j (exp2(G_last - G_j) dt_j) B_j (outer) x_j
// The running state h lives in tensor memory as an fp32 [s][p] accumulator
// (TMEM lane = s, column = p): each chunk the threads read it once (to store
// the start-of-chunk state as bf16 and to scale it by exp2(G_last)), write it
// back, and the chunk's tcgen05 MMAs accumulate the jump term onto it.
// Operands: TMA stages 64-token blocks of B (MN-major, s contiguous) and x
// (MN-major, p contiguous) three stages deep; the threads scale each x row by
// its weight in place.  The per-chunk states are written as bf16 in the
// layout [b, nh, nc, S, P] (p contiguous), which the output kernel loads by
// TMA as an MN-major operand; the final state is fp32 [b, nh, P, S].
#include "fwd.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 128;
constexpr int kKB = 64;   // tokens per pipeline stage
constexpr int kNST = 3;   // pipeline stages
constexpr int kBlk = kKB * 128;

__global__ void __launch_bounds__(kThreads)
fwd_state_bf16(const __grid_constant__ CUtensorMap tm_B, const __grid_constant__ CUtensorMap tm_x,
               const __nv_bfloat16 *__restrict__ dt, const float *__restrict__ A,
               const float *__restrict__ h0, __nv_bfloat16 *__restrict__ states,
               float *__restrict__ final_state, int *__restrict__ err, int L, int nh, int P,
               int S, int hpg, int T, int nc) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full[kNST], mmad[kNST];
  __shared__ uint32_t tmem_slot;
  __shared__ float Gs[256], w_s[256];
  __shared__ float warp_tot[4];

  constexpr int nMb = 2;  // 128 s = two 64-element (128-byte) blocks
  const int nPb = (P + 63) / 64;
  const int stage_bytes = (nMb + nPb) * kBlk;
  const int st_idx = blockIdx.x, h = blockIdx.y, b = blockIdx.z, g = h / hpg;
  const int s0 = st_idx * 128;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int srow = s0 + tid;  // this thread's state row (TMEM lane tid)
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const uint32_t ncols = P <= 32 ? 32 : (P <= 64 ? 64 : 128);
  const float Ah = A[h] * kLog2e;
  const int kbpc = T / kKB;
  const int nkb_last = (L - (nc - 1) * T + kKB - 1) / kKB;
  const int total_kb = (nc - 1) * kbpc + nkb_last;
  const int64_t bh = (int64_t)b * nh + h;

  if (tid == 0) {
    for (int i = 0; i < kNST; ++i) {
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
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;

  auto issue_loads = [&](int kbg) {
    const int st = kbg % kNST;
    const int k = kbg / kbpc, kb = kbg % kbpc;
    uint8_t *Ab = smem + st * stage_bytes;
    uint8_t *Xb = Ab + nMb * kBlk;
    const int tok = k * T + kb * kKB;
    ptx::mbar_arrive_expect_tx(&full[st], stage_bytes);
    for (int mb = 0; mb < nMb; ++mb)
      ptx::tma_load_4d(Ab + mb * kBlk, &tm_B, s0 + mb * 64, g, tok, b, &full[st]);
    for (int pb = 0; pb < nPb; ++pb)
      ptx::tma_load_4d(Xb + pb * kBlk, &tm_x, pb * 64, h, tok, b, &full[st]);
  };
  if (tid == 0)
    for (int i = 0; i < min(kNST, total_kb); ++i) issue_loads(i);

  // Chunk-local cumsum of A dt (log2 units) and the jump weights of chunk k.
  // Returns exp2(G_last).
  auto chunk_weights = [&](int k) -> float {
    const int valid = min(T, L - k * T);
    const int per = T > 128 ? 2 : 1;
    float d[2] = {0.f, 0.f}, c[2];
    float run = 0.f;
    for (int e = 0; e < per; ++e) {
      const int j = tid * per + e;
      if (j < valid) d[e] = __bfloat162float(dt[((int64_t)b * L + k * T + j) * nh + h]);
      run += Ah * d[e];
      c[e] = run;
    }
    float incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xffffffffu, incl, off);
      if ((tid & 31) >= off) incl += o;
    }
    if ((tid & 31) == 31) warp_tot[warp] = incl;
    __syncthreads();
    float base = incl - run;
    for (int w2 = 0; w2 < warp; ++w2) base += warp_tot[w2];
    for (int e = 0; e < per; ++e) {
      const int j = tid * per + e;
      if (j < T) Gs[j] = base + c[e];
    }
    __syncthreads();
    const float Glast = Gs[valid - 1];
    for (int e = 0; e < per; ++e) {
      const int j = tid * per + e;
      if (j < T) w_s[j] = j < valid ? exp2f(Glast - Gs[j]) * d[e] : 0.f;
    }
    __syncthreads();
    return exp2f(Glast);
  };

  // initial state into TMEM
  for (int c0 = 0; c0 < P; c0 += 16) {
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      v[j] = (h0 && srow < S) ? h0[(bh * P + c0 + j) * S + srow] : 0.f;
    ptx::tmem_st16(tmem + lane_base + c0, v);
  }
  ptx::tmem_st_wait();

  const uint32_t idesc = ptx::idesc_bf16(128, P, true, true);
  float gamma = chunk_weights(0);
  int kbg = 0;
  for (int k = 0; k < nc; ++k) {
    const int valid = min(T, L - k * T);
    const int nkb = (valid + kKB - 1) / kKB;
    if (k > 0) {
      const int last = kbg - 1;
      ptx::mbar_wait(&mmad[last % kNST], (last / kNST) & 1, err, 61);
      ptx::tc_fence_after();
    }
    // start of chunk k: store h (bf16, [s][p]) and scale it by exp2(G_last)
    __nv_bfloat16 *srow_out = states + ((bh * nc + k) * S + srow) * P;
    for (int c0 = 0; c0 < P; c0 += 16) {
      float v[16];
      ptx::tmem_ld16_sync(tmem + lane_base + c0, v);
      if (srow < S) {
        uint4 *o = reinterpret_cast<uint4 *>(srow_out + c0);
        o[0] = pack_io16(v, (__nv_bfloat16 *)nullptr);
        o[1] = pack_io16(v + 8, (__nv_bfloat16 *)nullptr);
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] *= gamma;
      ptx::tmem_st16(tmem + lane_base + c0, v);
    }
    ptx::tmem_st_wait();
    ptx::tc_fence_before();

    for (int kb = 0; kb < nkb; ++kb, ++kbg) {
      const int st = kbg % kNST;
      uint8_t *Ab = smem + st * stage_bytes;
      uint8_t *Xb = Ab + nMb * kBlk;
      ptx::mbar_wait(&full[st], (kbg / kNST) & 1, err, 62);
      for (int c = tid; c < nPb * kKB * 8; c += kThreads) {
        const float ws = w_s[kb * kKB + ((c >> 3) & (kKB - 1))];
        uint4 *p4 = reinterpret_cast<uint4 *>(Xb + c * 16);
        float v[8];
        unpack16(*p4, v, (__nv_bfloat16 *)nullptr);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] *= ws;
        *p4 = pack_op16(v, (__nv_bfloat16 *)nullptr);
      }
      ptx::fence_async_smem();
      __syncthreads();
      if (tid == 0) {
        ptx::tc_fence_after();
        const uint32_t a0 = ptx::smem_u32(Ab), x0 = ptx::smem_u32(Xb);
#pragma unroll
        for (int kk = 0; kk < kKB / 16; ++kk) {
          const uint64_t ad = ptx::smem_desc(a0 + kk * 2048, kBlk, 1024, ptx::kSw128);
          const uint64_t bd = ptx::smem_desc(x0 + kk * 2048, kBlk, 1024, ptx::kSw128);
          ptx::mma_ss<false>(tmem, ad, bd, idesc, 1u);
        }
        ptx::mma_commit(&mmad[st]);
        // refill the previous block's stage once its MMAs are done
        const int prev = kbg - 1;
        if (prev >= 0 && prev + kNST < total_kb) {
          ptx::mbar_wait(&mmad[prev % kNST], (prev / kNST) & 1, err, 63);
          issue_loads(prev + kNST);
        }
      }
    }
    if (k + 1 < nc) gamma = chunk_weights(k + 1);
  }
  {
    const int last = kbg - 1;
    ptx::mbar_wait(&mmad[last % kNST], (last / kNST) & 1, err, 64);
    ptx::tc_fence_after();
  }
  for (int c0 = 0; c0 < P; c0 += 16) {
    float v[16];
    ptx::tmem_ld16_sync(tmem + lane_base + c0, v);
    if (final_state && srow < S) {
#pragma unroll
      for (int j = 0; j < 16; ++j) final_state[(bh * P + c0 + j) * S + srow] = v[j];
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tmem, ncols);
}

}  // namespace

cudaError_t launch_fwd_state(const Dims &d, const void *x, const void *B, const void *dt,
                             const float *A, const float *h0, void *states, float *final_state,
                             cudaStream_t st) {
  CUtensorMap tB, tx;
  if (!make_tmap_bl(&tB, B, true, d.b, d.L, d.ng, d.S, kKB) ||
      !make_tmap_bl(&tx, x, true, d.b, d.L, d.nh, d.P, kKB))
    return cudaErrorInvalidValue;
  const int nPb = (int)((d.P + 63) / 64);
  const int smem = kNST * (2 + nPb) * kBlk + 1024;
  cudaError_t e =
      cudaFuncSetAttribute(fwd_state_bf16, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((d.S + 127) / 128), (unsigned)d.nh, (unsigned)d.b);
  fwd_state_bf16<<<grid, kThreads, smem, st>>>(
      tB, tx, static_cast<const __nv_bfloat16 *>(dt), A, h0,
      static_cast<__nv_bfloat16 *>(states), final_state, device_error_word(), (int)d.L,
      (int)d.nh, (int)d.P, (int)d.S, (int)d.hpg, (int)d.T, (int)d.nc);
  return cudaGetLastError();
}

}  // namespace ssd
