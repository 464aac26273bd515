// Host harness for the CUDA path's piece-start rules (tt_rules.cuh).
// Test infrastructure: it runs the SAME rule functions the kernels use, with
// the scans done sequentially, so the rules can be checked against the
// oracle on the CPU.  The parallel scans themselves are checked by the GPU
// parity tests.
#include <stdint.h>
#include <vector>
#include "../exact_bpe_tokenization_gb300/csrc/tt_rules.cuh"

using namespace tt;

// cp/raw/rs: per char of the whole batch (rs = first char of a request;
// deepseek-style raw kinds carry K_HAN_FLAG).  Writes 1/0 into start[] per
// char.
extern "C" void rules_host_starts(int fam, const uint32_t *cp, const uint8_t *raw, const uint8_t *rs_in, int64_t n,
                                  uint8_t *start) {
  // deepseek-style: the first two splitters' segment starts act as request starts
  std::vector<uint8_t> rsx(rs_in, rs_in + n);
  if (fam == FAM_DEEPSEEK)
    for (int64_t j = 1; j < n; ++j)
      if (ds_segment_start(raw[j - 1], raw[j])) rsx[j] = 1;
  const uint8_t *rs = rsx.data();
  std::vector<uint8_t> eff(n);
  // scan 1: mark resolution
  int64_t last_region = -1, last_trig = -1;
  for (int64_t j = 0; j < n; ++j) {
    uint8_t rp = (j > 0 && !rs[j]) ? raw[j - 1] : K_NONE;
    uint32_t cpp = (j > 0 && !rs[j]) ? cp[j - 1] : 0;
    uint8_t rn = (j + 1 < n && !rs[j + 1]) ? raw[j + 1] : K_NONE;
    if (region_start(raw[j], rp)) last_region = j;
    if (trigger(raw[j], rp, cpp, rn)) last_trig = j;
    bool mark_other = raw[j] == K_MARK && last_trig >= last_region && last_region >= 0;
    eff[j] = effective(fam, raw[j], mark_other);
  }
  std::vector<uint8_t> chain(n, 1);   // chain state after char j (inclusive)
  auto nbr = [&](int64_t j) {
    Nbr b;
    uint8_t *e[5] = {&b.e0, &b.e1, &b.e2, &b.e3, &b.e4};
    uint32_t *c[5] = {&b.c0, &b.c1, &b.c2, &b.c3, &b.c4};
    bool inside = true;
    for (int k = 0; k < 5; ++k) {
      int64_t x = j - k;
      if (k > 0 && (x < 0 || rs[x + 1])) inside = false;
      *e[k] = inside ? eff[x] : K_NONE;
      *c[k] = inside ? cp[x] : 0;
    }
    bool in1 = j + 1 < n && !rs[j + 1];
    bool in2 = in1 && j + 2 < n && !rs[j + 2];
    b.en1 = in1 ? eff[j + 1] : K_NONE;
    b.en2 = in2 ? eff[j + 2] : K_NONE;
    b.cn1 = in1 ? cp[j + 1] : 0;
    b.cn2 = in2 ? cp[j + 2] : 0;
    b.rs = rs[j] != 0;
    b.l1 = j >= 1 ? chain[j - 1] : true;
    b.l2 = j >= 2 ? chain[j - 2] : true;
    b.l3 = j >= 3 ? chain[j - 3] : true;
    return b;
  };
  // reverse queries (exclusive: first event strictly after j)
  std::vector<uint8_t> rq_ws(n), rq_up(n);
  uint8_t cw = R_END, cu = R_END;
  for (int64_t j = n - 1; j >= 0; --j) {
    rq_ws[j] = cw;
    rq_up[j] = cu;
    uint8_t ew = rq_ws_event(fam, rs[j], raw[j], cp[j]);
    uint8_t eu = rq_up_event(rs[j], raw[j]);
    if (ew != 0xFF) cw = ew;
    if (eu != 0xFF) cu = eu;
  }
  // forward scan (scan 2), sequential; chain states go into chain[] as we go.
  // The families without a case rule use the 12-byte state, as the kernels
  // do; both forms are run and must give the same aggregates.
  S2 before = s2_identity();
  S2L lbefore = s2l_identity();
  for (int64_t j = 0; j < n; ++j) {
    Nbr b = nbr(j);
    const S2 after = s2_trivial(fam, b) ? before
                     : s2_combine(before, s2_element(fam, b, (int32_t)j, (int32_t)(j + 1), (int32_t)(j + 2)));
    Aggs a;
    bool ch;
    s2_values(before, after, (int32_t)j, a, ch);
    chain[j] = ch;
    before = after;
    if (fam != FAM_O200K) {
      const S2L lafter = s2l_combine(lbefore, s2l_element(b.e0, b.e1, b.c0, (int32_t)j));
      Aggs la;
      s2l_values(lbefore, lafter, (int32_t)j, la);
      lbefore = lafter;
      if (b.e0 == K_NUM && la.nidx3 != a.nidx3) { start[j] = 2; continue; }          // 2: the forms disagree
      if (b.e0 == K_WS && (la.w_start != a.w_start || la.w_prev_other != a.w_prev_other ||
                           la.w_ncw_before != a.w_ncw_before)) { start[j] = 2; continue; }
      a = la;
    }
    a.rq_ws = rq_ws[j];
    a.rq_up = rq_up[j];
    start[j] = piece_start(fam, b, a) ? 1 : 0;
    if (fam != FAM_O200K && !needs_far_nbr(b.e0, b.e1)) {
      // the near fields alone decide: every other field scrambled
      Nbr nb = b;
      nb.e2 = nb.e3 = nb.e4 = (uint8_t)((j * 7 + 3) % 8);
      nb.c2 = nb.c3 = nb.c4 = (j & 1) ? (uint32_t)'\'' : (uint32_t)' ';
      nb.en2 = (uint8_t)((j * 5 + 1) % 8);
      nb.cn2 = (j & 2) ? (uint32_t)'s' : (uint32_t)'\n';
      nb.l1 = nb.l2 = nb.l3 = (j & 4) != 0;
      if ((piece_start(fam, nb, a) ? 1 : 0) != start[j]) start[j] = 3;   // 3: the near fields do not decide
    }
  }
}

// The kernels' gather of the top bit of each byte of a word.
extern "C" uint32_t rules_host_top_bits4(uint32_t w) { return top_bits4(w); }
