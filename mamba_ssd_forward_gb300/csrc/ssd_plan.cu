// Launch plans of the bf16 forward path: the candidates and the cost-model
// default.  Host code only, and stateless: a plan is passed to each call
// explicitly (or the default is used); the plans change launch shapes, never
// results.
#include "fwd.cuh"
#include "ssd_internal.cuh"

namespace ssd {

FwdPlan fwd_default_plan(const Dims &d) {
  FwdPlan p;
  p.cs = chunk_state_plan(d);
  if (fwd_out_supported(d)) {
    p.scan_kernel = 3;
    p.scan_heads = fwd_out_heads(d);
    return p;
  }
  p.scan_kernel = fwd_scan_chunk_supported(d) ? 1 : fwd_scan_chunk_split_supported(d) ? 2 : 0;
  p.scan_heads = p.scan_kernel ? fwd_scan_chunk_heads(d, p.scan_kernel == 2) : fwd_scan_heads(d);
  return p;
}

void fwd_cs_candidates(const Dims &d, std::vector<CsPlan> *out) {
  for (int ctas = 1; ctas <= 2; ++ctas)
    for (int H = 1; H <= 4; ++H)
      if (chunk_state_plan_ok(d, CsPlan{H, ctas})) out->push_back(CsPlan{H, ctas});
}

void fwd_scan_candidates(const Dims &d, std::vector<FwdPlan> *out) {
  FwdPlan p{};
  p.cs = CsPlan{0, 0};
  for (int hs = 1; hs <= d.hpg; ++hs)
    if (fwd_out_heads_ok(d, hs)) {
      p.scan_kernel = 3;
      p.scan_heads = hs;
      out->push_back(p);
    }
  for (int kind = 1; kind <= 2; ++kind)
    for (int hs = 1; hs <= d.hpg; ++hs)
      if (fwd_scan_chunk_heads_ok(d, hs, kind == 2)) {
        p.scan_kernel = kind;
        p.scan_heads = hs;
        out->push_back(p);
      }
  for (int H = 1; H <= 4; ++H)
    if (fwd_scan_heads_ok(d, H)) {
      p.scan_kernel = 0;
      p.scan_heads = H;
      out->push_back(p);
    }
}

bool fwd_plan_ok(const Dims &d, const FwdPlan &p) {
  if (!chunk_state_plan_ok(d, p.cs)) return false;
  if (p.scan_kernel == 1 || p.scan_kernel == 2)
    return fwd_scan_chunk_heads_ok(d, p.scan_heads, p.scan_kernel == 2);
  if (p.scan_kernel == 0) return fwd_scan_heads_ok(d, p.scan_heads);
  if (p.scan_kernel == 3) return fwd_out_heads_ok(d, p.scan_heads);
  return false;
}

}  // namespace ssd
