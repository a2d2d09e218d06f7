/*
 * Float64 CPU oracle for the Mamba-2 SSD forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * What it computes is the plain token-by-token recurrence, written out with
 * no chunking, blocking or reordering ("Accelerating Mamba-2 with
 * High-Performance Forward Pass Kernels in NVIDIA CUDA Tile",
 * section "Mamba-2 architecture", the core recurrence and its a_t/b_t form):
 *
 *     a_t = A[h] * dt_t
 *     H_t = exp(a_t) * H_{t-1} + (dt_t * x_t) (outer) B_t       (P x S)
 *     y_t = H_t . C_t + D[h] * x_t                              (P)
 *
 * Readings taken where the page is silent or garbled:
 *   - y uses the post-update state H_t (the causal mask of the page's
 *     linear-attention and chunked output equations keeps the diagonal);
 *   - x has headdim P entries and the state is stored P x S, the transpose
 *     of the page's S x H notation (the same page stores the initial and
 *     per-chunk states as [.., headdim, dstate] tiles);
 *   - heads share B and C by contiguous groups: g = h / (nheads / ngroups);
 *   - D is one scalar per head; a NULL D means D = 0, a NULL h0 means H = 0.
 *
 * Besides y and the final state it reports, per chunk of `chunk` tokens,
 * the quantities the four kernels of the page's decomposition hand to one
 * another, each by its plain definition:
 *   - G[b,h,k*T+i]: inclusive sum of a over tokens kT..kT+i of chunk k,
 *     natural-log units (the page stores it times log2(e)); positions past
 *     the end of the sequence hold the chunk's last real value (the page
 *     pads the partial last chunk with dt = 0);
 *   - states[b,h,k]: the recurrence state just before chunk k's first token
 *     (h0 for k = 0), as stored by the page's fwd_pass_state loop;
 *   - dstates[b,h,k]: the state reached by running the recurrence over chunk
 *     k's tokens alone, starting from zero.
 *
 * All tensors are dense row-major float64:
 *   x [b,L,nh,P]  dt [b,L,nh]  A [nh]  B,C [b,L,ng,S]  D [nh]
 *   h0, final_state [b,nh,P,S]  states, dstates [b,nh,nc,P,S]
 *   y [b,L,nh,P]  G [b,nh,nc*T]
 * `bh` (optional) lists flattened batch*nheads+head indices to compute;
 * outputs of other (b,h) pairs are left untouched.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

int ssd_oracle_forward(int64_t batch, int64_t seqlen, int64_t nheads,
                       int64_t headdim, int64_t dstate, int64_t ngroups,
                       int64_t chunk, const double *x, const double *dt,
                       const double *A, const double *B, const double *C,
                       const double *D, const double *h0, const int64_t *bh,
                       int64_t nbh, double *y, double *final_state,
                       double *states, double *dstates, double *G) {
  if (batch < 0 || seqlen < 0 || nheads <= 0 || headdim <= 0 || dstate <= 0 ||
      ngroups <= 0 || chunk <= 0 || nheads % ngroups != 0)
    return 1;
  const int64_t P = headdim, S = dstate, T = chunk;
  const int64_t nc = (seqlen + T - 1) / T;
  const int64_t hpg = nheads / ngroups;
  const int64_t npairs = bh ? nbh : batch * nheads;

  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t idx = 0; idx < npairs; ++idx) {
    const int64_t pair = bh ? bh[idx] : idx;
    if (pair < 0 || pair >= batch * nheads) {
      bad |= 1;
      continue;
    }
    const int64_t b = pair / nheads, h = pair % nheads, g = h / hpg;
    double *H = (double *)calloc((size_t)(P * S), sizeof(double));
    double *Hloc = (double *)calloc((size_t)(P * S), sizeof(double));
    if (!H || !Hloc) {
      free(H);
      free(Hloc);
      bad |= 2;
      continue;
    }
    if (h0)
      memcpy(H, h0 + pair * P * S, (size_t)(P * S) * sizeof(double));
    const double Dh = D ? D[h] : 0.0;
    double gsum = 0.0;

    for (int64_t t = 0; t < seqlen; ++t) {
      const int64_t k = t / T, i = t % T;
      if (i == 0) {
        /* start of chunk k: record the carried state, restart the chunk's
         * local state and its running log-decay */
        if (states)
          memcpy(states + (pair * nc + k) * P * S, H,
                 (size_t)(P * S) * sizeof(double));
        memset(Hloc, 0, (size_t)(P * S) * sizeof(double));
        gsum = 0.0;
      }
      const double dtv = dt[(b * seqlen + t) * nheads + h];
      const double a = A[h] * dtv;
      const double decay = exp(a);
      gsum += a;
      if (G) G[pair * nc * T + t] = gsum;

      const double *xt = x + ((b * seqlen + t) * nheads + h) * P;
      const double *Bt = B + ((b * seqlen + t) * ngroups + g) * S;
      const double *Ct = C + ((b * seqlen + t) * ngroups + g) * S;
      double *yt = y ? y + ((b * seqlen + t) * nheads + h) * P : NULL;
      for (int64_t p = 0; p < P; ++p) {
        const double u = dtv * xt[p];
        double *Hp = H + p * S;
        double acc = 0.0;
        for (int64_t s = 0; s < S; ++s) {
          Hp[s] = decay * Hp[s] + u * Bt[s];
          acc += Hp[s] * Ct[s];
        }
        if (yt) yt[p] = acc + Dh * xt[p];
        if (dstates) {
          double *Lp = Hloc + p * S;
          for (int64_t s = 0; s < S; ++s) Lp[s] = decay * Lp[s] + u * Bt[s];
        }
      }

      if (i == T - 1 || t == seqlen - 1) {
        /* end of chunk k: its local state is complete; pad G past the end
         * of the sequence with the last real value (dt = 0 there) */
        if (dstates)
          memcpy(dstates + (pair * nc + k) * P * S, Hloc,
                 (size_t)(P * S) * sizeof(double));
        if (G)
          for (int64_t j = t + 1; j < (k + 1) * T; ++j)
            G[pair * nc * T + j] = gsum;
      }
    }
    if (final_state)
      memcpy(final_state + pair * P * S, H, (size_t)(P * S) * sizeof(double));
    free(H);
    free(Hloc);
  }
  return bad;
}
