// Launch plans of the bf16 forward path: the candidates, the cost-model
// default, and the per-process table of installed plans that ssd_forward
// reads.  Host code only; the plans change launch shapes, never results.
#include <map>
#include <mutex>
#include <tuple>

#include "fwd.cuh"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

using Key = std::tuple<int, int64_t, int64_t, int64_t, int64_t, int64_t, int64_t, int64_t>;

std::mutex &table_mutex() {
  static std::mutex m;
  return m;
}
std::map<Key, FwdPlan> &table() {
  static std::map<Key, FwdPlan> t;
  return t;
}

bool key_of(const Dims &d, Key *k) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  *k = Key(dev, d.b, d.L, d.nh, d.P, d.S, d.ng, d.T);
  return true;
}

}  // namespace

FwdPlan fwd_default_plan(const Dims &d) {
  FwdPlan p;
  p.cs = chunk_state_plan(d);
  p.scan_kernel = fwd_scan_chunk_supported(d) ? 1 : fwd_scan_chunk_split_supported(d) ? 2 : 0;
  p.scan_heads = p.scan_kernel ? fwd_scan_chunk_heads(d, p.scan_kernel == 2) : fwd_scan_heads(d);
  return p;
}

FwdPlan fwd_current_plan(const Dims &d) {
  Key k;
  if (key_of(d, &k)) {
    std::lock_guard<std::mutex> g(table_mutex());
    const auto it = table().find(k);
    if (it != table().end()) return it->second;
  }
  return fwd_default_plan(d);
}

void fwd_cs_candidates(const Dims &d, std::vector<CsPlan> *out) {
  for (int ctas = 1; ctas <= 2; ++ctas)
    for (int H = 1; H <= 4; ++H)
      if (chunk_state_plan_ok(d, CsPlan{H, ctas})) out->push_back(CsPlan{H, ctas});
}

void fwd_scan_candidates(const Dims &d, std::vector<FwdPlan> *out) {
  FwdPlan p{};
  p.cs = CsPlan{0, 0};
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
  return false;
}

bool fwd_install_plan(const Dims &d, const FwdPlan *p) {
  Key k;
  if (!key_of(d, &k)) return false;
  std::lock_guard<std::mutex> g(table_mutex());
  if (p)
    table()[k] = *p;
  else
    table().erase(k);
  return true;
}

}  // namespace ssd
