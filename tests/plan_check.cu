// Host-only check of the single-token kernel's shared-memory plan
// (decode_plan_for), compiled and run by tests/test_plan_host.py.  For the
// shapes the tests and the bench use, and for random shapes inside the kernel's
// limits, every plan that is accepted must have: regions 128-byte aligned,
// disjoint and inside the total; the gate/up area holding the pre-routing
// pieces, the routed slices and the post-gate/up pieces (the down partials
// clear of the next layer's shared and router rows); every block's rows and
// copies inside their slots; and the lane and thread mappings covering every
// row.  Prints "ok <accepted> <rejected>" and exits 0, or names the first
// violation and exits 1.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "../bit_expert_matvec_moe_b300/csrc/moe_internal.h"

namespace {

int lo_row(int c, int P, int n) { return (int)((long long)c * n / P); }

struct Region {
  const char* name;
  size_t at, end;
};

bool check(int nsm, int optin, int H, int I, int E, int K, int bits, int sbits, int hs, int hg, bool* accepted) {
  moe::DecodePlan p;
  *accepted = moe::decode_plan_for(nsm, optin, H, I, E, K, bits, sbits, hs, hg, &p);
  if (!*accepted) return true;
  auto fail = [&](const char* what) {
    std::printf("plan H=%d I=%d E=%d K=%d bits=%d/%d hs=%d hg=%d: %s\n", H, I, E, K, bits, sbits, hs, hg, what);
    return false;
  };
  const int NE = K + hs, ngh = H / 64, ngi = I / 64;
  const moe::Fmt fr = moe::make_fmt(bits, H, I), fs = moe::make_fmt(hs ? sbits : bits, H, I);
  const size_t ngroups = std::max((size_t)NE * ngi, (size_t)ngh);
  // the gate/up area ends where the next region starts
  const size_t g_end = p.off_al;
  const size_t pre_end = std::max({p.off_sgu + (hs ? (size_t)p.rows_gu * fs.gu_pair : 0),
                                   p.off_rt + (size_t)p.rows_r * H * 2, p.off_hbuf + (size_t)H * 4});
  std::vector<Region> rs = {
      {"down slices", p.off_dn, p.off_dn + (size_t)NE * p.dn_slot},
      {"gate/up area", p.off_g, g_end},
      {"limbs", p.off_al, p.off_al + ngroups * moe::kLimbBytes},
      {"group factors", p.off_ae, p.off_ae + ngroups * 8},
      {"gate/up partials", p.off_part, p.off_part + (size_t)NE * p.part_stride * 4},
      {"router partials", p.off_rpart, p.off_rpart + (size_t)p.rows_r * moe::kWarps * 4},
      {"down sums", p.off_y, p.off_y + (size_t)p.rows_d * 4},
      {"mbarriers", p.off_bar, p.off_bar + (size_t)(1 + 2 * NE + 1) * 8},
      {"misc", p.off_misc, p.off_misc + 256 + 2 * sizeof(moe::DecodeLayer) + 32 * 4}};
  for (size_t i = 0; i < rs.size(); ++i) {
    if (rs[i].at % 128) return fail(rs[i].name);
    if (rs[i].end + 128 > p.total) return fail("region past the total");
    for (size_t j = i + 1; j < rs.size(); ++j)
      if (rs[i].at < rs[j].end && rs[j].at < rs[i].end) return fail("regions overlap");
  }
  const size_t gsz = g_end - p.off_g;
  if (pre_end > gsz) return fail("pre-routing pieces outside the gate/up area");
  if ((size_t)K * p.gu_slot > gsz) return fail("routed slices outside the gate/up area");
  const size_t pdn = (size_t)p.rows_d * NE * ngi * 4;
  if (p.off_pdn + pdn > gsz) return fail("down partials outside the gate/up area");
  // a stack launch copies the next layer's shared gate/up rows and router rows
  // while the down partials are in use
  const size_t next_end = std::max(p.off_sgu + (hs ? (size_t)p.rows_gu * fs.gu_pair : 0),
                                   p.off_rt + (size_t)p.rows_r * H * 2);
  if (p.off_pdn < next_end) return fail("down partials overlap the next layer's rows");
  if (p.off_sgu % 16 || p.off_rt % 16 || p.off_hbuf % 16 || p.gu_slot % 16 || p.dn_slot % 16)
    return fail("copy destination not 16-byte aligned");
  if (p.total > (size_t)optin) return fail("plan larger than the opt-in shared memory");
  for (int c = 0; c < p.P; ++c) {
    const int nr = lo_row(c + 1, p.P, I) - lo_row(c, p.P, I);
    const int nj = lo_row(c + 1, p.P, H) - lo_row(c, p.P, H);
    const int nrr = lo_row(c + 1, p.P, E) - lo_row(c, p.P, E) + (hg && c == 0 ? 1 : 0);
    if (nr > p.rows_gu || nj > p.rows_d || nrr > p.rows_r) return fail("block rows beyond the plan");
    if ((size_t)nr * fr.gu_pair > p.gu_slot || (size_t)nj * std::max(fr.d_row, fs.d_row) > p.dn_slot)
      return fail("block copy beyond its slot");
  }
  // lane and thread mappings: gate/up (2 rows per lane stream), down (set, unit)
  // with up to 5 rows per thread, router / SwiGLU rows by one warp, row sums by
  // 16 threads per row
  const moe::RowMap mh = moe::make_rowmap(ngh);
  if (2 * (moe::kWarps / mh.chunks) * mh.rpp < 2 * p.rows_gu) return fail("gate/up rows not covered");
  const int Q = NE * ngi, S = moe::kBlock / Q;
  if (S < 1 || 5 * S < p.rows_d) return fail("down rows not covered");
  if (p.rows_gu > 32 || p.rows_r > 32 || p.rows_d * 16 > moe::kBlock) return fail("one-warp / row-sum limits");
  return true;
}

}  // namespace

int main() {
  const int nsm = 148, optin = 232448;
  struct S {
    int H, I, E, K, bits, sbits, hs, hg;
  };
  std::vector<S> shapes = {{4096, 1024, 512, 4, 4, 4, 1, 0}, {4096, 1024, 512, 4, 4, 4, 1, 1},
                           {4096, 1024, 512, 4, 2, 4, 1, 0}, {4096, 1024, 512, 4, 2, 2, 1, 0},
                           {4096, 1024, 64, 4, 4, 4, 1, 0},  {4096, 1024, 512, 4, 4, 4, 0, 0},
                           {256, 128, 16, 4, 4, 4, 1, 0},    {256, 128, 16, 4, 4, 4, 1, 1},
                           {256, 128, 16, 4, 4, 4, 0, 0},    {256, 128, 4, 4, 4, 4, 1, 0},
                           {256, 128, 16, 1, 4, 4, 1, 0},    {320, 64, 24, 3, 4, 4, 1, 0},
                           {256, 128, 16, 4, 2, 2, 1, 0},    {256, 128, 16, 8, 4, 4, 1, 0},
                           {256, 128, 16, 2, 4, 4, 1, 0},    {2048, 768, 128, 8, 4, 4, 0, 0},
                           {64, 64, 1, 1, 4, 4, 0, 0},       {256, 128, 16, 4, 2, 4, 1, 1}};
  // the full-width layer must take the single-token kernel
  int acc = 0, rej = 0;
  for (size_t i = 0; i < shapes.size(); ++i) {
    const S& s = shapes[i];
    bool ok = false;
    if (!check(nsm, optin, s.H, s.I, s.E, s.K, s.bits, s.sbits, s.hs, s.hg, &ok)) return 1;
    if (i < 5 && !ok) {
      std::printf("full-width shape %zu rejected by the plan\n", i);
      return 1;
    }
    (ok ? acc : rej)++;
  }
  std::srand(20260101);
  for (int it = 0; it < 3000; ++it) {
    const int H = 64 * (1 + std::rand() % 64), I = 64 * (1 + std::rand() % 32);
    const int E = 1 + std::rand() % 1024, K = 1 + std::rand() % std::min(8, E);
    const int bits = std::rand() % 2 ? 4 : 2, sbits = std::rand() % 2 ? 4 : 2;
    const int hs = std::rand() % 2, hg = hs && std::rand() % 2;
    bool ok = false;
    if (!check(nsm, optin, H, I, E, K, bits, sbits, hs, hg, &ok)) return 1;
    (ok ? acc : rej)++;
  }
  std::printf("ok %d %d\n", acc, rej);
  return 0;
}
