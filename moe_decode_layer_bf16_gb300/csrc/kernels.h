// Internal launch interfaces between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kBlock = 128;  // weight scale block side / activation group length

// Header words at the start of a moe_decode_layer workspace (int32 each).
enum HdrWord {
  kHdrStatus = 0,        // 0 or MOE_ERR_DEVICE_TIMEOUT (sticky until read)
  kHdrFault = 1,         // test hook: withhold the first slot's ready signal
  kHdrRouterTicket = 2,  // router CTAs whose logits are complete
  kHdrQueue = 3,         // expert-kernel work queue head
  kHdrActive = 4,        // number of routed experts with at least one route
  kHdrDoneA = 5,         // w13 items finished (h stored and, when due, its group quantised)
  kHdrXReady = 6,        // router CTAs that have quantised their share of x (and, CTA 0, reset
                         // the expert kernel's counters); the expert kernel's last CTA clears it
  kHdrExit = 7,          // expert-kernel CTAs finished
  kHdrRouterFin = 8,     // router CTAs that have routed their share of the tokens
  kHdrWords = 64
};
constexpr int kMaxRouterTickets = 1024;
constexpr int kMaxMk = 4096;       // M * top_k per call
constexpr int kMaxTokens = 4096;   // M per call (the bound for a dense layer, whose top_k is 0)
constexpr int kMaxExperts = 512;
constexpr int kMaxTopK = 16;

// Stream-K split of a skinny GEMM Y[M, N] = A[M, K] . W[N, K]^T over G CTAs.
// Work cells are (token chunk, 64-row tile, 128-column k-block), k fastest;
// CTA c owns cells [c*T/G, (c+1)*T/G).
// With dyn_tiles > 0 the last dyn_tiles (chunk, tile)s are left out of the
// static split: they are cut into units of dyn_unit k-blocks (dyn_nu a tile,
// fixed boundaries) that the CTAs take from a counter once their static share
// is done, so that the CTAs that stream faster take the tail.
struct GemvPlan {
  int M, N, K;
  int chunk_tokens;  // 8, 16 or 32
  int n_chunks, n_tiles, nkb;
  long long total;   // statically split cells
  int G;             // CTAs
  int max_segs;      // most static runs that cover one (chunk, tile)
  int dyn_tiles = 0, dyn_unit = 0, dyn_nu = 0;
};
void plan_gemv(GemvPlan& p, int M, int N, int K, int G, int dyn_tiles = 0);
// (chunk, tile)s of the dynamic tail of an automatic split-K plan over n_ct
// of them, and its unit length in k-blocks
inline long long splitk_dyn_tiles(long long n_ct) { return n_ct >= 32 ? n_ct / 8 : 0; }
constexpr int kDynUnit = 4;
constexpr int kDynMinRun = 64;  // static cells a CTA streams at least for the tail to be used
// resident CTAs per SM of the split-K (router == false) or router kernel on
// the current device (cached per device)
int gemv_blocks_per_sm(int chunk_tokens, bool router);
size_t gemv_partials_bytes(const GemvPlan& p);
// token chunk of a skinny GEMM of M tokens: 8, 16 or 32 columns per CTA pass
inline int gemv_chunk_tokens(int M) { return M <= 8 ? 8 : (M <= 16 ? 16 : 32); }

// SM count of the current device (cached per device): MOE_OK or MOE_ERR_CUDA.
int current_device_sms(int* sms);
// The plan of one split-K projection, shared by every entry point that runs
// it.  split_k == 0: stream-K over all SMs (every CTA streams an equal share
// of W); split_k = S > 0: every (token chunk, 64-row tile) is cut into exactly
// S K-segments, one CTA each.  Returns MOE_OK, MOE_ERR_INVALID_ARG or
// MOE_ERR_UNSUPPORTED (shape or split out of range) or MOE_ERR_CUDA.
int plan_splitk(GemvPlan& p, int M, int N, int K, int split_k);
// Bytes of the plan's counters (one per (chunk, tile), then the dynamic
// tail's unit counter and exit counter; rounded up to 256) and of its partial
// sums (0 when no tile is split).
size_t splitk_ticket_bytes(const GemvPlan& p);
size_t splitk_partial_bytes(const GemvPlan& p);

struct SplitKArgs {
  const void* A;
  const void* W;
  void* C;
  int c_fp32;
  float alpha;
  float* partials;
  unsigned* tickets;
  // programmatic dependent launch: the kernel starts while the preceding one
  // (which writes A, never W) ends, prefetches its first weights into L2 and
  // waits for that kernel before it reads A
  bool pdl = false;
};
cudaError_t launch_splitk(const GemvPlan& p, const SplitKArgs& a, cudaStream_t s);

struct RouterArgs {
  const void* x;       // bf16 [M, H]
  const void* W;       // bf16 [E, H]
  const float* bias;   // [E] or null
  int E, k, e8m0;
  float scaling;
  float* partials;
  unsigned* tickets;
  float* logits;       // [M, E]
  uint8_t* xq;         // [M, H]
  float* xs;           // [M, H/128]
  int* hdr;
  int* ids;            // [M*k]
  float* tw;           // [M*k]
  int* sorted;         // [M*k]
  int* off;            // [E+1]
  int* act;            // [E]
  int* gcount;         // expert-kernel counters reset here
  int n_gcount;
  int* ready;
  int n_ready;
  int32_t* user_ids;
  float* user_w;
  int32_t* user_sorted;
  int32_t* user_off;
};
cudaError_t launch_router(const GemvPlan& p, const RouterArgs& a, cudaStream_t s);

struct ExpertArgs {
  int H, I, Is, E, k, M, Mk, Imax, gI;
  int hsS;  // row stride (floats) of the h scales: gI rounded up to 32 (one 128-byte line per row)
  float limit;
  int e8m0;
  const uint8_t* w13; const float* w13_s;
  const uint8_t* w2;  const float* w2_s;
  const uint8_t* sw13; const float* sw13_s;
  const uint8_t* sw2;  const float* sw2_s;
  const uint8_t* xq; const float* xs;
  const int* sorted; const int* off; const int* act;
  int* hdr; int* gcount; int* ready;
  float* h; uint8_t* hq; float* hs;
  float* rows; float* shared_out;
  int router_ctas;  // CTAs of the router launch that precedes this kernel
  int bq;           // w2 item size in 32-row quarters of a 128-row block: 4, 2 or 1
};
// An expert-kernel launch prepared on the host (tensor maps encoded, the
// pass width and ring depth chosen, the shared-memory limit set) before the
// router is enqueued, so that no host work falls between the router's and the
// expert kernel's launches.
// Extra arguments of the tensor-core (tcgen05) form of the expert kernel:
//   xg       the routed tokens' x codes in route order (launch_gather_rows)
//   sh_segs  K segments of the shared slot's w2 items (tc_shared_segments),
//            whose partial rows follow one another in shared_out
//   a_segs   K segments of the shared slot's w13 items (tc_w13_segments),
//            partial [g; u] rows in gu_part (tc_w13_partial_bytes), counted
//            per group in pcount (zeroed by the router with the counters)
struct TcExtra {
  const uint8_t* xg;
  int sh_segs;
  int a_segs;
  float* gu_part;
  int* pcount;
};
struct ExpertsLaunch {
  ExpertArgs a;
  CUtensorMap maps[7];
  bool tc;               // the tcgen05 kernel (else the warp-MMA kernel)
  int tt;                // warp-MMA kernel: 8-token columns per pass
  int nst;               // warp-MMA kernel: ring stages
  size_t smem;           // dynamic shared memory
  TcExtra tcx;           // tcgen05 kernel
};
cudaError_t prepare_experts(const ExpertArgs& a, ExpertsLaunch& L);
cudaError_t prepare_experts_tc(const ExpertArgs& a, const TcExtra& x, ExpertsLaunch& L);
cudaError_t launch_experts(const ExpertsLaunch& L, int num_sms, cudaStream_t s);
cudaError_t launch_gather_rows(const uint8_t* xq, const int* sorted, int k, int Mk, int H, uint8_t* xg, int num_sms,
                               cudaStream_t s);
constexpr int kMaxSharedSegs = 16;  // K segments of a dense layer's w2 items at most
int tc_shared_segments(int E, int H, int Is, int M, int num_sms);
int tc_w13_segments(int E, int H, int Is, int M);
size_t tc_w13_partial_bytes(int E, int Is);

struct NormArgs {
  const void* x; const void* residual; const void* gain;
  const float* rows; const float* route_w; const float* shared;
  void* out; void* residual_out;
  int M, H, k;
  int shared_parts;  // partial rows [parts][M][H] in `shared`, added in order (>= 1)
  float* m_out;      // non-null: write m (fp32 [M, H]) there and stop (no residual, no norm)
  float eps;
  int early;  // residual and gain come from before the preceding kernels (the layer call)
};
cudaError_t launch_rmsnorm(const NormArgs& a, cudaStream_t s);

struct EhNormArgs {
  const int32_t* ids; const void* embed; int vocab;
  const void* hidden; const void* enorm; const void* hnorm;
  float eps;
  void* out;  // bf16 [M, 2H]
  int M, H;
  int* status;
};
cudaError_t launch_eh_norm(const EhNormArgs& a, cudaStream_t s);

// Launch configuration that lets a kernel start while its predecessor in the
// stream finishes (it waits with griddepcontrol.wait before using its results).
struct PdlLaunch {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  PdlLaunch(dim3 grid, dim3 block, size_t smem, cudaStream_t s) {
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
};

}  // namespace moe
