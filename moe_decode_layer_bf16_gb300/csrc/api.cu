// C ABI of libmoe_decode.so (declared in include/moe_decode.h): argument
// checks, workspace layout and kernel launches.  Host code only.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>

#include "../../include/moe_decode.h"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kGemvMaxCtas = 2048;

size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Bytes of the stream-K partial sums for any grid of at most kGemvMaxCtas
// CTAs: nkb contiguous cells meet at most ceil(nkb / shortest run) + 1 runs.
size_t gemv_partials_bound(int M, int N, int K) {
  GemvPlan p;
  p.chunk_tokens = gemv_chunk_tokens(M);
  p.n_chunks = (M + p.chunk_tokens - 1) / p.chunk_tokens;
  p.n_tiles = (N + 63) / 64;
  p.nkb = K / kBlock;
  const long long total = (long long)p.n_chunks * p.n_tiles * p.nkb;
  // every CTA's run is at least floor(total / G) >= floor(total / kGemvMaxCtas) cells long
  const long long minrun = std::max<long long>(1, total / kGemvMaxCtas);
  p.max_segs = (int)std::min<long long>(p.nkb, (p.nkb + minrun - 1) / minrun + 1);
  return gemv_partials_bytes(p);
}

// The same bound for an automatic split-K plan, with or without the dynamic
// tail: a static split over all tiles, or over all but the tail's tiles
// (shorter runs) with the tail tiles' units.
size_t splitk_partials_bound(int M, int N, int K) {
  GemvPlan p;
  p.chunk_tokens = gemv_chunk_tokens(M);
  p.n_chunks = (M + p.chunk_tokens - 1) / p.chunk_tokens;
  p.n_tiles = (N + 63) / 64;
  p.nkb = K / kBlock;
  const long long n_ct = (long long)p.n_chunks * p.n_tiles;
  p.dyn_tiles = (int)splitk_dyn_tiles(n_ct);
  p.dyn_nu = p.dyn_tiles > 0 ? (p.nkb + std::min(kDynUnit, p.nkb) - 1) / std::min(kDynUnit, p.nkb) : 0;
  const long long total = (n_ct - p.dyn_tiles) * p.nkb;
  const long long minrun = std::max<long long>(1, total / kGemvMaxCtas);
  p.max_segs = (int)std::min<long long>(p.nkb, (p.nkb + minrun - 1) / minrun + 1);
  return std::max(gemv_partials_bytes(p), gemv_partials_bound(M, N, K));
}

struct Layout {
  size_t hdr, tickets, gcount, ready, partials, logits, xq, xs, ids, tw, sorted, off, act;
  size_t h, hq, hs, rows, shared, xg, gu_part, total;
  int n_gcount, n_ready, Imax, gI, hsS;
};

// Rows of the shared output region for M tokens: the tensor-core kernel may
// split a dense layer's w2 items into K segments (partial rows the boundary
// adds) while one pass holds all tokens; bounded so that the region grows
// with M.
size_t shared_rows(const moe_layer_dims& d, int M) {
  // (at most kMaxSharedSegs segments, whatever the SM count)
  const int segs = std::max(1, std::min(kMaxSharedSegs, d.shared_inter / kBlock));
  return (size_t)std::max<long long>(M, (long long)(d.num_experts == 0 ? segs : 1) * std::min(M, 64));
}

// Which expert kernel a call runs (moe_set_expert_path overrides the choice):
// the tensor-core kernel where the tokens of an expert can make a real
// contraction (a dense layer from 4 tokens, an MoE layer from 16 tokens:
// measured on the DeepSeek-V3-shaped layers, where below these counts the
// warp-MMA kernel's finer items start the routed w2 work sooner), else the
// warp-MMA kernel.
std::atomic<int> g_path_override{0};

int expert_path(const moe_layer_dims& d, int M) {
  const int o = g_path_override.load(std::memory_order_relaxed);
  if (o == MOE_PATH_WARP_MMA || o == MOE_PATH_TCGEN05) return o;
  if (d.num_experts == 0) return M >= 4 ? MOE_PATH_TCGEN05 : MOE_PATH_WARP_MMA;
  return M >= 16 ? MOE_PATH_TCGEN05 : MOE_PATH_WARP_MMA;
}

void layout_for(const moe_layer_dims& d, int M, Layout& L) {
  const int H = d.hidden, E = d.num_experts, k = d.top_k;
  L.Imax = std::max(d.inter, d.shared_inter);
  L.gI = L.Imax / kBlock;
  L.hsS = (L.gI + 31) / 32 * 32;
  L.n_gcount = 2 * (E + 1) * L.gI;  // the expert kernels' group counters, then the split-segment counts
  L.n_ready = E + 1;
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o = align_up(o + bytes); return at; };
  L.hdr = take(kHdrWords * sizeof(int));
  L.tickets = take(kMaxRouterTickets * sizeof(unsigned));
  L.gcount = take((size_t)L.n_gcount * sizeof(int));
  L.ready = take((size_t)L.n_ready * sizeof(int));
  L.partials = take(gemv_partials_bound(M, E, H));
  L.logits = take((size_t)M * E * sizeof(float));
  L.xq = take((size_t)M * H);
  L.xs = take((size_t)M * (H / kBlock) * sizeof(float));
  L.ids = take((size_t)M * k * sizeof(int));
  L.tw = take((size_t)M * k * sizeof(float));
  L.sorted = take((size_t)M * k * sizeof(int));
  L.off = take((size_t)(E + 1) * sizeof(int));
  L.act = take((size_t)E * sizeof(int));
  const size_t hrows = (size_t)M * k + M;
  L.h = take(hrows * L.Imax * sizeof(float));
  L.hq = take(hrows * L.Imax);
  L.hs = take(hrows * L.hsS * sizeof(float));
  L.rows = take((size_t)M * k * H * sizeof(float));
  L.shared = take(shared_rows(d, M) * H * sizeof(float));
  L.xg = take((size_t)M * k * H);
  L.gu_part = take(tc_w13_partial_bytes(E, d.shared_inter));
  L.total = o;
}

int check_dims(const moe_layer_dims* d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->num_experts == 0) {
    // a dense layer: the MLP in the shared-expert slot, no router, no routed experts
    if (d->top_k != 0 || d->inter != 0 || d->shared_inter <= 0) return MOE_ERR_INVALID_ARG;
  } else if (d->inter <= 0 || d->top_k <= 0) {
    return MOE_ERR_INVALID_ARG;
  }
  if (d->hidden <= 0 || d->shared_inter < 0 || d->num_experts < 0) return MOE_ERR_INVALID_ARG;
  if (!std::isfinite(d->routed_scaling) || !(d->swiglu_limit > 0.f) || !(d->rms_eps >= 0.f) ||
      !std::isfinite(d->rms_eps))
    return MOE_ERR_INVALID_ARG;
  if (d->hidden % kBlock || d->hidden > 16384) return MOE_ERR_UNSUPPORTED;
  if (d->inter % kBlock || d->inter > 8192) return MOE_ERR_UNSUPPORTED;
  if (d->shared_inter % kBlock || d->shared_inter > 32768) return MOE_ERR_UNSUPPORTED;
  if (d->num_experts > kMaxExperts || d->num_experts % 16) return MOE_ERR_UNSUPPORTED;
  if (d->top_k > kMaxTopK || d->top_k > d->num_experts) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int gemv_grid(long long cells, int sms, int per_sm) {
  return (int)std::max<long long>(1, std::min<long long>({cells, (long long)sms * per_sm, (long long)kGemvMaxCtas}));
}

int check_splitk_shape(int M, int N, int K, int split_k) {
  if (M < 1 || N < 1 || K < 1 || split_k < 0) return MOE_ERR_INVALID_ARG;
  if (M > 256 || N % 16 || K % kBlock) return MOE_ERR_UNSUPPORTED;
  if (split_k > K / kBlock) return MOE_ERR_UNSUPPORTED;  // at most one k-block per segment
  return MOE_OK;
}

long long tiles_of(int M, int N) {
  const int chunk = gemv_chunk_tokens(M);
  return (long long)((M + chunk - 1) / chunk) * ((N + 63) / 64);
}

}  // namespace

// Host threads may make their first calls at the same time: the cached values
// are atomics (a race only computes the same value twice).
int current_device_sms(int* out) {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (!n) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return MOE_ERR_CUDA;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  *out = n;
  return MOE_OK;
}

int plan_splitk(GemvPlan& plan, int M, int N, int K, int split_k) {
  int rc = check_splitk_shape(M, N, K, split_k);
  if (rc != MOE_OK) return rc;
  const long long n_ct = tiles_of(M, N);
  long long G;
  if (split_k > 0) {
    // CTA c owns cells [c T / G, (c + 1) T / G) with T = n_ct * nkb and
    // G = n_ct * S: the runs start at every tile's first k-block and cut
    // each tile into exactly S segments
    G = n_ct * split_k;
    if (G > INT_MAX) return MOE_ERR_UNSUPPORTED;
  } else {
    int sms = 0;
    if ((rc = current_device_sms(&sms)) != MOE_OK) return rc;
    G = gemv_grid(n_ct * (K / kBlock), sms, gemv_blocks_per_sm(gemv_chunk_tokens(M), false));
  }
  // The dynamic tail pays where every CTA streams a long static share (each
  // unit starts its loads cold: measured, LM head at 1.85 GB 299 -> 276 us,
  // eh_proj at 205 MB 40.9 -> 41.4 us); an explicit split keeps every segment
  // where it was asked for.
  const bool tail = split_k == 0 && n_ct * (K / kBlock) >= kDynMinRun * G;
  plan_gemv(plan, M, N, K, (int)G, tail ? (int)splitk_dyn_tiles(n_ct) : 0);
  return MOE_OK;
}

size_t splitk_ticket_bytes(const GemvPlan& p) {
  return align_up(((size_t)p.n_chunks * p.n_tiles + 2) * sizeof(unsigned));
}

size_t splitk_partial_bytes(const GemvPlan& p) {
  return p.max_segs > 1 || p.dyn_nu > 1 ? gemv_partials_bytes(p) : 0;
}

// splitk_gemm_bf16 with the launch form: pdl lets the kernel start while the
// preceding kernel of the stream, which writes A (never W), still runs.
int splitk_impl(const void* A, const void* W, void* C, int c_fp32, int M, int N, int K, int split_k, float alpha,
                void* ws, size_t ws_bytes, void* stream, bool pdl) {
  size_t need = 0;
  int rc = splitk_gemm_workspace_size(M, N, K, split_k, &need);
  if (rc != MOE_OK) return rc;
  if (!A || !W || !C || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(W) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
  GemvPlan plan;
  if ((rc = plan_splitk(plan, M, N, K, split_k)) != MOE_OK) return rc;
  const size_t tickets = splitk_ticket_bytes(plan);
  if (tickets + splitk_partial_bytes(plan) > need) return MOE_ERR_UNSUPPORTED;
  SplitKArgs a;
  a.A = A; a.W = W; a.C = C; a.c_fp32 = c_fp32 ? 1 : 0; a.alpha = alpha;
  a.tickets = reinterpret_cast<unsigned*>(ws);
  a.partials = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + tickets);
  a.pdl = pdl;
  return launch_splitk(plan, a, (cudaStream_t)stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_decode_workspace_size(const moe_layer_dims* dims, int max_tokens, size_t* bytes) {
  const int rc = check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (!bytes || max_tokens < 1) return MOE_ERR_INVALID_ARG;
  if (max_tokens > kMaxTokens || (long long)max_tokens * dims->top_k > kMaxMk) return MOE_ERR_UNSUPPORTED;
  Layout L;
  layout_for(*dims, max_tokens, L);
  *bytes = L.total;
  return MOE_OK;
}

int moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  return cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

static int layer_impl(const moe_layer_dims* dims, const moe_layer_weights* w, int M, const void* x,
                      const void* residual, void* out, void* residual_out, int32_t* topk_ids,
                      float* topk_w, int32_t* sorted_routes, int32_t* expert_offsets, void* workspace,
                      size_t ws_bytes, void* stream, void* const* events, float* m_out = nullptr) {
  int rc = check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (!w || M < 0) return MOE_ERR_INVALID_ARG;
  if (M == 0) return MOE_OK;
  if (M > kMaxTokens || (long long)M * dims->top_k > kMaxMk) return MOE_ERR_UNSUPPORTED;
  const bool has_shared = dims->shared_inter > 0;
  const bool dense = dims->num_experts == 0;  // routed weights are not read (may be NULL)
  if (!dense && (!w->router_w || !w->w13 || !w->w13_s || !w->w2 || !w->w2_s)) return MOE_ERR_INVALID_ARG;
  const bool partial = m_out != nullptr;  // a rank's partial sum: no residual, gain or outputs
  if (!partial && !w->norm_gain) return MOE_ERR_INVALID_ARG;
  if (has_shared && (!w->sw13 || !w->sw13_s || !w->sw2 || !w->sw2_s)) return MOE_ERR_INVALID_ARG;
  if (!x || !workspace || (!partial && (!residual || !out || !residual_out))) return MOE_ERR_INVALID_ARG;
  if ((!dense && (!aligned16(w->router_w) || !aligned16(w->w13) || !aligned16(w->w2))) || !aligned16(x) ||
      !aligned16(workspace) || (has_shared && (!aligned16(w->sw13) || !aligned16(w->sw2))) ||
      (partial ? !aligned16(m_out)
               : (!aligned16(residual) || !aligned16(out) || !aligned16(residual_out) || !aligned16(w->norm_gain))))
    return MOE_ERR_INVALID_ARG;
  Layout L;
  layout_for(*dims, M, L);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  int sms = 0;
  if ((rc = current_device_sms(&sms)) != MOE_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  const int H = dims->hidden, E = dims->num_experts, k = dims->top_k;

  GemvPlan plan;
  const int chunk = gemv_chunk_tokens(M);
  const long long cells = (long long)((M + chunk - 1) / chunk) * ((E + 63) / 64) * (H / kBlock);
  // at least 2 (M <= 8) or 4 k-blocks per CTA: shorter runs start the routing
  // sooner at one token chunk, more partial sums to add cost more above (measured)
  const int run = M <= 8 ? 2 : 4;
  plan_gemv(plan, M, E, H, gemv_grid((cells + run - 1) / run, sms, gemv_blocks_per_sm(chunk, true)));
  if (dense) {
    // no logits: the router kernel only quantises x (one warp per 1024-column
    // slice of a token, 4 warps a CTA) and resets the expert kernel's counters
    const long long slices = (long long)M * ((H / kBlock + 7) / 8);
    plan.G = (int)std::max<long long>(1, std::min<long long>((slices + 3) / 4, sms));
  }
  if ((long long)plan.n_chunks * plan.n_tiles > kMaxRouterTickets) return MOE_ERR_UNSUPPORTED;
  if (gemv_partials_bytes(plan) > gemv_partials_bound(M, E, H)) return MOE_ERR_UNSUPPORTED;

  RouterArgs ra;
  ra.x = x; ra.W = w->router_w; ra.bias = w->sel_bias; ra.E = E; ra.k = k; ra.e8m0 = dims->e8m0 ? 1 : 0;
  ra.scaling = dims->routed_scaling;
  ra.partials = reinterpret_cast<float*>(ws + L.partials);
  ra.tickets = reinterpret_cast<unsigned*>(ws + L.tickets);
  ra.logits = reinterpret_cast<float*>(ws + L.logits);
  ra.xq = ws + L.xq;
  ra.xs = reinterpret_cast<float*>(ws + L.xs);
  ra.hdr = reinterpret_cast<int*>(ws + L.hdr);
  ra.ids = reinterpret_cast<int*>(ws + L.ids);
  ra.tw = reinterpret_cast<float*>(ws + L.tw);
  ra.sorted = reinterpret_cast<int*>(ws + L.sorted);
  ra.off = reinterpret_cast<int*>(ws + L.off);
  ra.act = reinterpret_cast<int*>(ws + L.act);
  ra.gcount = reinterpret_cast<int*>(ws + L.gcount);
  ra.n_gcount = L.n_gcount;
  ra.ready = reinterpret_cast<int*>(ws + L.ready);
  ra.n_ready = L.n_ready;
  ra.user_ids = topk_ids; ra.user_w = topk_w; ra.user_sorted = sorted_routes; ra.user_off = expert_offsets;
  ExpertArgs ea;
  ea.H = H; ea.I = dims->inter; ea.Is = dims->shared_inter; ea.E = E; ea.k = k; ea.M = M; ea.Mk = M * k;
  ea.Imax = L.Imax; ea.gI = L.gI; ea.hsS = L.hsS;
  ea.limit = dims->swiglu_limit; ea.e8m0 = dims->e8m0 ? 1 : 0;
  ea.w13 = w->w13; ea.w13_s = w->w13_s; ea.w2 = w->w2; ea.w2_s = w->w2_s;
  ea.sw13 = w->sw13; ea.sw13_s = w->sw13_s; ea.sw2 = w->sw2; ea.sw2_s = w->sw2_s;
  ea.xq = ra.xq; ea.xs = ra.xs; ea.sorted = ra.sorted; ea.off = ra.off; ea.act = ra.act;
  ea.hdr = ra.hdr; ea.gcount = ra.gcount; ea.ready = ra.ready;
  ea.h = reinterpret_cast<float*>(ws + L.h);
  ea.hq = ws + L.hq;
  ea.hs = reinterpret_cast<float*>(ws + L.hs);
  ea.rows = reinterpret_cast<float*>(ws + L.rows);
  ea.shared_out = reinterpret_cast<float*>(ws + L.shared);
  ea.router_ctas = plan.G;
  // a w2 item streams its 32-row groups over all of I: 4 of them (a whole
  // scale block) unless the rows are long (I >= 8192, a dense layer's MLP),
  // where single groups keep the queue's tail short, or the whole-block items
  // would give the SMs no more than 4 each (one token's 8 experts and the
  // shared one: 504 items over 152 SMs), where half blocks even out the tail
  const long long w2_items = (std::min<long long>((long long)M * k, E) + (dims->shared_inter > 0 ? 1 : 0)) * (H / kBlock);
  ea.bq = L.Imax >= 8192 ? 1 : (w2_items <= 4LL * sms ? 2 : 4);
  // every expert-kernel launch parameter is prepared before the router is
  // enqueued, so that no host work delays the expert kernel behind it
  const bool tc = expert_path(*dims, M) == MOE_PATH_TCGEN05;
  uint8_t* xg = ws + L.xg;
  const int parts = tc ? tc_shared_segments(E, H, dims->shared_inter, M, sms) : 1;
  // the partial rows of split w2 items must fit the shared-output region
  if ((size_t)parts * M > shared_rows(*dims, M)) return MOE_ERR_UNSUPPORTED;
  TcExtra tx;
  tx.xg = xg;
  tx.sh_segs = parts;
  tx.a_segs = tc_w13_segments(E, H, dims->shared_inter, M);
  tx.gu_part = reinterpret_cast<float*>(ws + L.gu_part);
  tx.pcount = ea.gcount + (E + 1) * L.gI;
  ExpertsLaunch el;
  if ((tc ? prepare_experts_tc(ea, tx, el) : prepare_experts(ea, el)) != cudaSuccess) return MOE_ERR_CUDA;
  auto mark = [&](int i) {
    return !events || cudaEventRecord((cudaEvent_t)events[i], s) == cudaSuccess;
  };
  if (!mark(0)) return MOE_ERR_CUDA;
  if (launch_router(plan, ra, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (!mark(1)) return MOE_ERR_CUDA;
  // routed tokens' x rows in route order first (only the routing is waited for)
  if (tc && !dense && launch_gather_rows(ra.xq, ra.sorted, k, M * k, H, xg, sms, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_experts(el, sms, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (!mark(2)) return MOE_ERR_CUDA;

  NormArgs na;
  na.x = nullptr; na.residual = residual; na.gain = w->norm_gain;
  na.rows = ea.rows; na.route_w = ra.tw; na.shared = has_shared ? ea.shared_out : nullptr;
  na.shared_parts = parts;
  na.m_out = m_out;
  na.out = out; na.residual_out = residual_out; na.M = M; na.H = H; na.k = k; na.eps = dims->rms_eps;
  // the residual and the gain were written before the router's plain launch,
  // so the boundary may load them before it waits on the expert kernel
  na.early = 1;
  if (launch_rmsnorm(na, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (!mark(3)) return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_decode_layer(const moe_layer_dims* dims, const moe_layer_weights* w, int M, const void* x,
                     const void* residual, void* out, void* residual_out, int32_t* topk_ids,
                     float* topk_w, int32_t* sorted_routes, int32_t* expert_offsets, void* workspace,
                     size_t ws_bytes, void* stream) {
  return layer_impl(dims, w, M, x, residual, out, residual_out, topk_ids, topk_w, sorted_routes,
                    expert_offsets, workspace, ws_bytes, stream, nullptr);
}

int moe_decode_layer_traced(const moe_layer_dims* dims, const moe_layer_weights* w, int M, const void* x,
                            const void* residual, void* out, void* residual_out, int32_t* topk_ids,
                            float* topk_w, int32_t* sorted_routes, int32_t* expert_offsets,
                            void* workspace, size_t ws_bytes, void* stream, void* const* events) {
  if (!events || !events[0] || !events[1] || !events[2] || !events[3]) return MOE_ERR_INVALID_ARG;
  return layer_impl(dims, w, M, x, residual, out, residual_out, topk_ids, topk_w, sorted_routes,
                    expert_offsets, workspace, ws_bytes, stream, events);
}

int moe_decode_layer_partial(const moe_layer_dims* dims, const moe_layer_weights* w, int M, const void* x,
                             float* m_out, int32_t* topk_ids, float* topk_w, int32_t* sorted_routes,
                             int32_t* expert_offsets, void* workspace, size_t ws_bytes, void* stream) {
  if (!m_out && M > 0) return MOE_ERR_INVALID_ARG;  // (M == 0 returns before any pointer is used)
  return layer_impl(dims, w, M, x, nullptr, nullptr, nullptr, topk_ids, topk_w, sorted_routes, expert_offsets,
                    workspace, ws_bytes, stream, nullptr, m_out);
}

int moe_tp_boundary(const float* partials, int G, const void* residual, const void* gain, int M, int H, float eps,
                    void* out, void* residual_out, void* stream) {
  if (M < 0 || H <= 0 || G < 1 || !(eps >= 0.f)) return MOE_ERR_INVALID_ARG;
  if (H % kBlock || H > 16384) return MOE_ERR_UNSUPPORTED;
  if (!partials || !residual || !gain || !out || !residual_out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(partials) || !aligned16(residual) || !aligned16(gain) || !aligned16(out) || !aligned16(residual_out))
    return MOE_ERR_INVALID_ARG;
  if (M == 0) return MOE_OK;
  NormArgs na;
  na.x = nullptr; na.residual = residual; na.gain = gain; na.rows = nullptr; na.route_w = nullptr;
  na.shared = partials; na.shared_parts = G; na.m_out = nullptr;
  na.out = out; na.residual_out = residual_out; na.M = M; na.H = H; na.k = 0; na.eps = eps;
  na.early = 0;  // the partials may come from the kernel just before
  return launch_rmsnorm(na, (cudaStream_t)stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int splitk_gemm_workspace_size(int M, int N, int K, int split_k, size_t* bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARG;
  const int rc = check_splitk_shape(M, N, K, split_k);
  if (rc != MOE_OK) return rc;
  const long long n_ct = tiles_of(M, N);
  // the automatic split depends on the device's SM count: its bound covers any grid
  const size_t partials = split_k == 0 ? splitk_partials_bound(M, N, K)
                          : split_k == 1 ? 0
                                         : (size_t)n_ct * split_k * gemv_chunk_tokens(M) * 64 * sizeof(float);
  *bytes = align_up(((size_t)n_ct + 2) * sizeof(unsigned)) + partials;
  return MOE_OK;
}

int splitk_gemm_bf16(const void* A, const void* W, void* C, int c_fp32, int M, int N, int K, int split_k,
                     float alpha, void* ws, size_t ws_bytes, void* stream) {
  return splitk_impl(A, W, C, c_fp32, M, N, K, split_k, alpha, ws, ws_bytes, stream, false);
}

int rmsnorm_residual(const void* x, const void* residual, const void* gain, int M, int H, float eps,
                     const float* rows, const float* route_w, int k, const float* shared, void* out,
                     void* residual_out, void* stream) {
  if (M < 0 || H <= 0 || !(eps >= 0.f)) return MOE_ERR_INVALID_ARG;
  if (H % kBlock || H > 16384) return MOE_ERR_UNSUPPORTED;
  if (!residual || !gain || !out || !residual_out) return MOE_ERR_INVALID_ARG;
  if (rows && (!route_w || k < 1 || k > kMaxTopK)) return MOE_ERR_INVALID_ARG;
  if ((x && !aligned16(x)) || !aligned16(residual) || !aligned16(gain) || !aligned16(out) ||
      !aligned16(residual_out) || (rows && !aligned16(rows)) || (shared && !aligned16(shared)))
    return MOE_ERR_INVALID_ARG;
  if (M == 0) return MOE_OK;
  NormArgs na;
  na.x = x; na.residual = residual; na.gain = gain; na.rows = rows; na.route_w = route_w;
  na.shared = shared; na.shared_parts = 1; na.m_out = nullptr; na.out = out; na.residual_out = residual_out;
  na.M = M; na.H = H;
  na.k = rows ? k : 0; na.eps = eps;
  na.early = 0;  // the preceding kernel may be the one that writes them
  return launch_rmsnorm(na, (cudaStream_t)stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// MTP front workspace: a 256-byte header (status word), A = bf16 [M, 2H], then
// the split-K tickets and partial sums of the eh_proj projection.
constexpr size_t kMtpHdr = 256;

int mtp_eh_front_workspace_size(int M, int H, size_t* bytes) {
  if (!bytes || M < 1 || H < 1) return MOE_ERR_INVALID_ARG;
  if (M > 256 || H % kBlock || H > 16384) return MOE_ERR_UNSUPPORTED;
  size_t gemm = 0;
  const int rc = splitk_gemm_workspace_size(M, H, 2 * H, 0, &gemm);
  if (rc != MOE_OK) return rc;
  *bytes = kMtpHdr + align_up((size_t)M * 2 * H * 2) + gemm;
  return MOE_OK;
}

int mtp_eh_front(const int32_t* input_ids, const void* embed, int vocab, const void* hidden, const void* enorm,
                 const void* hnorm, float eps, const void* eh_proj_w, int M, int H, void* out, void* ws,
                 size_t ws_bytes, void* stream) {
  size_t need = 0;
  int rc = mtp_eh_front_workspace_size(M, H, &need);
  if (rc != MOE_OK) return rc;
  if (vocab < 1 || !(eps >= 0.f)) return MOE_ERR_INVALID_ARG;
  if (!input_ids || !embed || !hidden || !enorm || !hnorm || !eh_proj_w || !out || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned16(embed) || !aligned16(hidden) || !aligned16(enorm) || !aligned16(hnorm) || !aligned16(eh_proj_w) ||
      !aligned16(out) || !aligned16(ws))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* w = reinterpret_cast<uint8_t*>(ws);
  void* A = w + kMtpHdr;
  uint8_t* gemm_ws = w + kMtpHdr + align_up((size_t)M * 2 * H * 2);
  EhNormArgs ea;
  ea.ids = input_ids; ea.embed = embed; ea.vocab = vocab; ea.hidden = hidden; ea.enorm = enorm; ea.hnorm = hnorm;
  ea.eps = eps; ea.out = A; ea.M = M; ea.H = H;
  ea.status = reinterpret_cast<int*>(w) + kHdrStatus;
  if (launch_eh_norm(ea, (cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
  // the projection's weights stream while the norm kernel still runs
  return splitk_impl(A, eh_proj_w, out, 0, M, H, 2 * H, 0, 1.f, gemm_ws, need - (gemm_ws - w), stream, true);
}

int moe_set_expert_path(int path) {
  if (path != MOE_PATH_AUTO && path != MOE_PATH_WARP_MMA && path != MOE_PATH_TCGEN05) return MOE_ERR_INVALID_ARG;
  g_path_override.store(path, std::memory_order_relaxed);
  return MOE_OK;
}

int moe_decode_layer_plan(const moe_layer_dims* dims, int M, int* path, int* launches) {
  const int rc = check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (M < 0 || !path || !launches) return MOE_ERR_INVALID_ARG;
  if (M > kMaxTokens || (long long)M * dims->top_k > kMaxMk) return MOE_ERR_UNSUPPORTED;
  *path = M == 0 ? MOE_PATH_AUTO : expert_path(*dims, M);
  *launches = M == 0 ? 0 : (*path == MOE_PATH_TCGEN05 && dims->num_experts > 0 ? 4 : 3);
  return MOE_OK;
}

int moe_device_status(void* ws, void* stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  int st = 0;
  if (cudaMemcpy(&st, reinterpret_cast<int*>(ws) + kHdrStatus, sizeof(int), cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaMemset(reinterpret_cast<int*>(ws) + kHdrStatus, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  return st;
}

int moe_debug_set_fault(void* ws, int fault, void* stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  const int v = fault ? 1 : 0;
  if (cudaMemcpy(reinterpret_cast<int*>(ws) + kHdrFault, &v, sizeof(int), cudaMemcpyHostToDevice) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

const char* moe_status_str(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_SCRATCH_LIMIT: return "problem exceeds the static scratch of the no-allocation entry point";
    default: return "unknown status";
  }
}

}  // extern "C"
