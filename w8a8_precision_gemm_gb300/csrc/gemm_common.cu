// gemm_common.cu -- tile planning and the split-K reduction of the W8A8 GEMM.
#include <algorithm>

#include "gemm.cuh"

namespace qurl {

// Decode (M <= 256, and INT8 at any M given the workspace): weights on the MMA
// M side, tokens padded to a power of two >= 16 on the N side (<= 256 for FP8,
// <= 128 for INT8, whose TMEM also holds the widened weights).  FP8 prefill and
// INT8 prefill without workspace: 128-token tiles x 256 (FP8) or 128 (INT8)
// channels.  When the tiles do not fill the SMs, K is split
// so that tiles x splits is close to the SM count, each split at least 512
// deep, as far as the workspace allows.  Workspace layout: [fp16 activation
// codes and per-token sums of |code| (INT8 decode)][split-K partials].
// INT8 prefill from this many tokens on: CTA pairs with both operands widened
// to fp16 in the workspace (the weights' widening, 3 N K bytes of HBM traffic,
// costs ~425 / M of the GEMM's tensor time).  Below it the TMEM-operand
// kernels are faster (measured on the 32B-class shapes at M = 512 and 1024),
// except their CTA-pair form, whose chunked accumulation runs two half passes
// over the weights: where the planner would pick that form, the widened kernel
// takes its place (gate_up at M = 1024: 447-453 us against 399 us with small
// activation codes and 780 us with normed ones).
constexpr int kWideMinM = 2048;
constexpr int kAttachedMinM = 256;

// The INT8 plan on CTA pairs with widened operands, when the workspace holds it.
bool plan_wide(GemmPlan& p, int M, int N, int K, int num_sms, size_t ws_avail, bool w_attached) {
  auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  p = GemmPlan{};
  p.wide = true;
  p.pair = true;
  p.swap = false;
  p.bn = 256;
  p.bk = 64;
  p.num_kb = (K + 63) / 64;
  p.tiles_tok = (M + 255) / 256;
  p.tiles_ch = (N + 255) / 256;
  const long long tiles = static_cast<long long>(p.tiles_tok) * p.tiles_ch;
  const int slots = std::max(1, num_sms / 2);
  // K splits (ranges of a multiple of 4 k-blocks, 256 codes: the code sums' granularity) only when the
  // pair tiles leave the pairs mostly idle
  const int cap = std::max(1, std::min(p.num_kb / 16, kMaxSums));
  int splits = 1;
  if (tiles < slots) splits = std::max(1, std::min(static_cast<int>(slots / tiles), cap));
  // k-blocks per split for s splits (a multiple of 4: the code sums' granularity)
  auto kps_of = [&](int s) { return ((p.num_kb + s - 1) / s + 3) & ~3; };
  // Rough time of s splits, as for the other kernels: rounds of units over
  // the pairs x (k-blocks per unit + pipeline fill and drain) x one 64-deep
  // k-block of a 256 x 256 unit at the fp16 rate (0.33 us), plus the
  // reduction (launch, s fp32/int32 partials read, bf16 written).  Taken over
  // the rule above when predicted 10% faster: shapes whose units fill a last
  // round of pairs barely.
  auto est = [&](int s) {
    const int kps = kps_of(s);
    const int ns = (p.num_kb + kps - 1) / kps;
    const double rounds = static_cast<double>((tiles * ns + slots - 1) / slots);
    double t = rounds * (kps + 9) * 0.33;
    if (ns > 1) t += 3.0 + (static_cast<double>(ns) * M * N * 4 + static_cast<double>(M) * N * 2) / 4e6;
    return t;
  };
  {
    const double t_rule = est(splits);
    int best = splits;
    double t_best = t_rule;
    for (int s = 1; s <= std::min(cap, 64); ++s) {
      const double t = est(s);
      if (t < t_best) {
        t_best = t;
        best = s;
      }
    }
    if (t_best < 0.9 * t_rule) splits = best;
  }
  // Hybrid: when whole-K units would leave a last round of pairs mostly idle
  // (tiles a little above a multiple of the pairs), the tiles of that last
  // round alone are split so that their pieces fill it, and a reduction kernel
  // finishes only them.  Taken over the plan above when the model says it
  // saves 3% and 8 us (below that the first round's start-up, which the model
  // leaves out, ate the gain: 32B qkv at M = 1024, predicted 4 us faster,
  // measured 1 us slower).  Measured: 32B o_proj at M = 1024, 76 whole + 4
  // tiles split five ways, 60.6 us a call against 64.9; 32B down at M = 8192,
  // 608 whole + 32 split two ways, 1169 us against 1212.
  int whole = 0;
  if (tiles > slots && tiles % slots != 0) {
    const double t_cur = est(splits);
    const long long rem = tiles % slots;
    const int st = std::min(static_cast<int>(slots / rem), cap);
    if (st >= 2) {
      const int kps_t = kps_of(st);
      const int ns = (p.num_kb + kps_t - 1) / kps_t;
      const double unit = (p.num_kb + 9) * 0.33;
      const double t_hyb = static_cast<double>(tiles / slots) * unit +
                           static_cast<double>((rem * ns + slots - 1) / slots) * (kps_t + 9) * 0.33 + 3.0 +
                           static_cast<double>(rem) * 65536.0 * (4.0 * ns + 2.0) / 4e6;
      if (t_hyb < 0.97 * t_cur && t_cur - t_hyb > 8.0) {
        whole = static_cast<int>(tiles - rem);
        splits = ns;
      }
    }
  }
  p.whole_units = whole;
  int kps = kps_of(splits);
  splits = (p.num_kb + kps - 1) / kps;
  const size_t x16 = al(static_cast<size_t>(M) * K * 2);
  const size_t sums = al(static_cast<size_t>(M) * 4 * splits);
  // weights attached by the caller (their fp16 copy and sums live in the caller's buffer)
  const size_t w16 = w_attached ? 0 : al(static_cast<size_t>(N) * K * 2);
  const size_t qn = w_attached ? 0 : al(static_cast<size_t>(N) * 4);
  const size_t scratch = static_cast<size_t>(i8w_max_ctas(num_sms)) * 256 * 128 * 4;
  const size_t part = splits > 1 ? static_cast<size_t>(splits) * M * N * 4 : 0;
  p.kb_per_split = kps;
  p.splits = splits;
  p.asum_off = x16;
  p.qsum_off = x16 + sums;
  p.w16_off = p.qsum_off + sums;
  p.qn_off = p.w16_off + w16;
  p.scratch_off = p.qn_off + qn;
  p.x16_bytes = p.scratch_off + scratch;  // everything before the split-K partials
  p.part_bytes = part;
  p.ws_bytes = p.x16_bytes + part;
  return p.ws_bytes <= ws_avail;
}

GemmPlan plan_narrow(int M, int N, int K, int qt, int num_sms, size_t ws_avail);

bool plan_nvfp4(GemmPlan& p, int M, int N, int K, int num_sms, size_t ws_avail, bool w_attached) {
  return plan_wide(p, M, N, K, num_sms, ws_avail, w_attached);
}

// INT8 whose weights' fp16 copy the caller keeps (qurl_widen_weights): the
// CTA-pair kernel above kAttachedMinM tokens, and from kAttachedBigMinM tokens
// for weights of at least kAttachedBigCodes codes.  It reads 2 bytes a weight,
// so for the smaller projections at up to 256 tokens the TMEM-weight kernel,
// which streams the 1-byte codes, is faster (32B-class qkv / o_proj at
// M = 256: 28.5 / 27.8 us against 35.4 / 32.9; 7B qkv 23.5 against 27.3);
// for the large ones the pair kernel's full-rate 256 x 256 tiles win even half
// empty (M = 256: 32B gate_up 109.6 against 125.9, down 79.8 against 88.5, 7B
// gate_up 59.5 against 65.6, down 53.4 against 54.2; gate_up at M = 160 105.8
// against 126.3), and above 256 tokens for every projection (M = 1024: qkv 69
// -> 64 us, o_proj 68 -> 63, down 285 -> 273).
constexpr int kAttachedBigMinM = 129;
constexpr long long kAttachedBigCodes = 1LL << 26;

bool plan_attached(GemmPlan& p, int M, int N, int K, int num_sms, size_t ws_avail) {
  const bool big = M >= kAttachedBigMinM && static_cast<long long>(N) * K >= kAttachedBigCodes;
  if ((M <= kAttachedMinM && !big) || ws_avail < kSyncBytes) return false;
  if (!plan_wide(p, M, N, K, num_sms, ws_avail - kSyncBytes, true)) return false;
  p.ws_bytes += kSyncBytes;
  return true;
}

GemmPlan plan_data(int M, int N, int K, int qt, int num_sms, size_t ws_avail) {
  GemmPlan w{};
  if (qt == kQInt8 && M >= kWideMinM && plan_wide(w, M, N, K, num_sms, ws_avail, false)) return w;
  const GemmPlan p = plan_narrow(M, N, K, qt, num_sms, ws_avail);
  if (p.tmem_a && p.pair && plan_wide(w, M, N, K, num_sms, ws_avail, false)) return w;
  return p;
}

// The last kSyncBytes of every workspace are reserved for the handoff counters
// of the fused entry points; the plan's regions fit before them.
GemmPlan plan_gemm(int M, int N, int K, int qt, int num_sms, size_t ws_avail) {
  GemmPlan p = plan_data(M, N, K, qt, num_sms, ws_avail >= kSyncBytes ? ws_avail - kSyncBytes : 0);
  p.ws_bytes += kSyncBytes;
  return p;
}

// The plans without widened weights: TMEM-operand INT8 kernels, FP8, and the
// shared-memory INT8 kernel.
GemmPlan plan_narrow(int M, int N, int K, int qt, int num_sms, size_t ws_avail) {
  GemmPlan p{};
  const bool int8 = (qt == kQInt8);
  // INT8 prefers the TMEM-operand kernel (weights on the MMA M side at every
  // M), which needs an fp16 copy of the activation codes (2 M K bytes) and
  // their sums in the workspace; without it, INT8 widens both operands in
  // shared memory.
  const size_t x16 = (static_cast<size_t>(M) * K * 2 + 255) & ~static_cast<size_t>(255);
  auto sums = [&](int s) { return (static_cast<size_t>(M) * 4 * s + 255) & ~static_cast<size_t>(255); };
  // the running sums of chunked units, one 128 x 128 int32 region per CTA
  const size_t scratch = static_cast<size_t>(std::max(num_sms, 1)) * 128 * 128 * 4;
  p.tmem_a = int8 && ws_avail >= x16 + sums(1) + scratch;
  p.swap = p.tmem_a || M <= 256;
  p.bk = int8 ? (p.tmem_a ? 256 : 64) : 128;
  p.num_kb = (K + p.bk - 1) / p.bk;
  if (p.swap) {
    const int max_bn = (int8 && !p.tmem_a) ? 128 : 256;
    int bn = 16;
    while (bn < M && bn < max_bn) bn *= 2;
    // CTA pairs (256 channels per pair) when there is enough work, at least
    // 1024 stages of pair tiles (stages of 128 bytes of K for FP8, 256 for
    // INT8; measured slower on the small qkv / o_proj, where half as many
    // tiles need more K splits): FP8 beyond 64 tokens (7B gate_up and down
    // at M = 256), INT8 beyond 256 tokens with 256-token tiles (prefill; in
    // the decode chain at M = 256 the single-CTA kernel, whose accumulator is
    // double-buffered and which overlaps the quantizer before it, measured
    // as fast)
    const long long pair_work = static_cast<long long>((M + (p.tmem_a ? 255 : bn - 1)) / (p.tmem_a ? 256 : bn)) *
                                ((N + 255) / 256) * p.num_kb;
    // INT8 pairs also need to fill their waves: a round of 256 x 256 units on
    // the SM pairs takes ~1.8 rounds of 128 x 128 units on the SMs (measured on
    // 7B gate_up, M = 4096), so the pairs are taken only when they need fewer
    // rounds by that factor (e.g. not for 32B qkv at M = 1024: 112 pair units
    // fill two rounds of 76 pairs half-way, 448 single units three rounds)
    bool pair_waves = true;
    if (p.tmem_a && bn == 256 && num_sms >= 2) {
      const long long up = static_cast<long long>((M + 255) / 256) * ((N + 255) / 256);
      const long long us = static_cast<long long>((M + 127) / 128) * ((N + 127) / 128);
      const long long rp = (up + num_sms / 2 - 1) / (num_sms / 2), rs = (us + num_sms - 1) / num_sms;
      pair_waves = 18 * rp <= 10 * rs;
    }
    if (p.tmem_a && bn == 256 && (pair_work < 1024 || M <= 256 || !pair_waves)) bn = 128;  // single-CTA tiles
    p.bn = bn;
    p.tiles_tok = (M + bn - 1) / bn;
    p.pair = pair_work >= 1024 && ((p.tmem_a && bn == 256) || (!int8 && bn >= 128));
    p.tiles_ch = p.pair ? (N + 255) / 256 : (N + 127) / 128;
  } else {
    p.bn = int8 ? 128 : 256;
    // FP8 prefill runs on CTA pairs: 256 tokens x 256 channels per pair
    p.pair = !int8;
    p.tiles_tok = (M + (p.pair ? 255 : 127)) / (p.pair ? 256 : 128);
    p.tiles_ch = (N + p.bn - 1) / p.bn;
  }
  const long long tiles = static_cast<long long>(p.tiles_tok) * p.tiles_ch;
  // units run one per SM, or one per SM pair
  const int slots = p.pair ? num_sms / 2 : num_sms;
  const int min_kb = (p.bk == 64) ? 8 : (p.bk == 256 ? 2 : 4);
  const int cap = std::max(1, std::min(p.num_kb / min_kb, p.tmem_a ? kMaxSums : 1 << 20));
  int splits = 1;
  if (slots > 0 && tiles < slots) splits = std::max(1, std::min(static_cast<int>(slots / tiles), cap));
  if (slots > 0) {
    // Rough time of s splits: rounds of units over the SMs x (k-blocks per
    // unit + a fixed pipeline fill and drain), plus the reduction kernel
    // (launch, reading s partials, writing the output).  A split count is
    // taken over the rule above only when it is predicted 10% faster: this
    // fixes shapes whose tiles leave a wave mostly empty (e.g. 320 tiles on
    // 152 SMs), and leaves the rest alone.
    const double stage_us = p.tmem_a ? (p.bn >= 128 ? 0.95 : 0.8) : (p.swap ? 0.36 : 0.45);
    const double fill = p.tmem_a ? 3.0 : 5.0;
    auto est = [&](int s) {
      const int kps = (p.num_kb + s - 1) / s;
      const int ns = (p.num_kb + kps - 1) / kps;
      const double rounds = static_cast<double>((tiles * ns + slots - 1) / slots);
      double t = rounds * (kps + fill) * stage_us;
      if (ns > 1) t += 3.0 + (static_cast<double>(ns) * M * N * 4 + static_cast<double>(M) * N * 2) / 4e6;
      return t;
    };
    const double t_rule = est(splits);
    int best = splits;
    double t_best = t_rule;
    for (int s = 1; s <= std::min(cap, 64); ++s) {
      const double t = est(s);
      if (t < t_best) {
        t_best = t;
        best = s;
      }
    }
    if (t_best < 0.9 * t_rule) splits = best;
    // FP8 prefill on CTA pairs: whole-K units plus a split tail, as for the
    // INT8 prefill kernel, when the last round of pair units would be mostly
    // idle and the model saves 3% and 15 us (32B down at M = 1024: 80 tiles on
    // 76 pairs, 76 whole + 4 split 18 ways, 93 us a call against 124 with K
    // split four ways; 32B o_proj at M = 1024, predicted 10 us faster, measured
    // 3 us slower: the few units of a last round run faster alone than the
    // model's shared rate says, more so for short K)
    if (!int8 && p.pair && !p.swap && tiles > slots && tiles % slots != 0) {
      const double t_cur = est(splits);
      const long long rem = tiles % slots;
      const int st = std::min(static_cast<int>(slots / rem), cap);
      if (st >= 2) {
        const int kps_t = (p.num_kb + st - 1) / st;
        const int ns = (p.num_kb + kps_t - 1) / kps_t;
        const double unit = (p.num_kb + fill) * stage_us;
        const double t_hyb = static_cast<double>(tiles / slots) * unit +
                             static_cast<double>((rem * ns + slots - 1) / slots) * (kps_t + fill) * stage_us + 3.0 +
                             static_cast<double>(rem) * 65536.0 * (4.0 * ns + 2.0) / 4e6;
        if (t_hyb < 0.97 * t_cur && t_cur - t_hyb > 15.0) {
          p.whole_units = static_cast<int>(tiles - rem);
          splits = ns;
        }
      }
    }
  }
  const size_t per_split = static_cast<size_t>(M) * N * 4;
  // workspace for s splits: [fp16 codes, code sums (INT8 decode)][s partials if s > 1]
  auto need = [&](int s) {
    return (p.tmem_a ? x16 + sums(s) + scratch : 0) + (s > 1 ? static_cast<size_t>(s) * per_split : 0);
  };
  while (splits > 1 && need(splits) > ws_avail) --splits;
  if (splits == 1) p.whole_units = 0;
  p.kb_per_split = (p.num_kb + splits - 1) / splits;
  p.splits = (p.num_kb + p.kb_per_split - 1) / p.kb_per_split;
  p.x16_bytes = p.tmem_a ? x16 + sums(p.splits) + scratch : 0;
  p.asum_off = p.tmem_a ? x16 : 0;
  p.scratch_off = p.tmem_a ? x16 + sums(p.splits) : 0;
  p.part_bytes = p.splits > 1 ? static_cast<size_t>(p.splits) * per_split : 0;
  p.ws_bytes = p.x16_bytes + p.part_bytes;
  return p;
}

int persistent_ctas(const GemmArgs& a) {
  static int sms[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  int n = (dev >= 0 && dev < 64) ? sms[dev] : 0;
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    if (dev >= 0 && dev < 64) sms[dev] = n;
  }
  const long long units = static_cast<long long>(a.tiles_tok) * a.tiles_ch * a.splits;
  return static_cast<int>(std::max<long long>(1, std::min<long long>(units, n)));
}

cudaError_t launch_splitk_reduce(int qt, const void* part, int splits, int M, int N, const float* sx,
                                 const float* sw, void* Y, long long ldy, void* acc_out, int num_sms,
                                 cudaStream_t st) {
  const size_t total = static_cast<size_t>(M) * N;
  const size_t items = (N % 4 == 0) ? total / 4 : total;
  size_t blocks = (items + 255) / 256;
  blocks = std::min<size_t>(blocks, static_cast<size_t>(num_sms > 0 ? num_sms : 152) * 8);
  blocks = std::max<size_t>(blocks, 1);
  auto* y = reinterpret_cast<__nv_bfloat16*>(Y);
  if (qt == kQInt8)
    return launch_pdl(splitk_reduce_kernel<int>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st,
                      reinterpret_cast<const int*>(part), splits, M, N, sx, sw, y, ldy,
                      reinterpret_cast<int*>(acc_out));
  return launch_pdl(splitk_reduce_kernel<float>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st,
                    reinterpret_cast<const float*>(part), splits, M, N, sx, sw, y, ldy,
                    reinterpret_cast<float*>(acc_out));
}

}  // namespace qurl
