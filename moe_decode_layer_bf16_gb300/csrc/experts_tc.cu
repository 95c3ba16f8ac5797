// The routed + shared experts of one decode step on the 5th-generation tensor
// cores, for steps whose experts hold many tokens: the decode page's grouped
// form (vllm.models.glm5next.nvidia.specialized_decode.runtime.decode,
// LayerStages._build_mega builds GroupedExperts for the larger token counts,
// and the grouped kernel runs the shared expert as one more expert), and dense
// layers (LayerStages._build_dense: the dense MLP's FP8 GEMMs) above a few
// tokens.  It computes exactly what experts.cu computes:
//   [g; u] = xq . w13^T with 128x128 block scales, h = silu(min(g, L)) *
//   clamp(u, -L, L), h quantised to FP8 per token per 128 intermediates,
//   y = hq . w2^T,
// routed rows unweighted in expanded route order, the shared expert's rows
// apart (a dense layer's long w2 rows split over K into partial rows that the
// boundary adds).
//
// Where experts.cu runs warp-level MMAs on 8- or 16-token passes, this kernel
// issues tcgen05.mma.kind::f8f6f4 (E4M3 x E4M3, fp32 accumulators in tensor
// memory) on passes of up to 64 tokens, so that the instruction count per
// weight byte no longer grows with the tokens of a pass:
//   * one CTA per SM, 12 warps: a producer warp (TMA), an MMA warp (one
//     thread issues every MMA and owns the tensor memory), two idle warps and
//     eight epilogue warps (two per tensor-memory lane quadrant, 32 token
//     columns each);
//   * work items from one atomic queue, all w13 items (shared expert first)
//     before all w2 items:
//       A item (expert, 128 intermediates): 128 gate + 128 up rows of w13
//       over H, i.e. one whole 128-column group of h;
//       B item (expert, 128 rows of w2, one K segment of I): 128 rows;
//     each runs once per pass of <= 64 of the expert's tokens;
//   * a stage holds two (weight tile, activation tile) pairs in 128-byte
//     swizzled K-major layout: A items one k-block of the gate and the up
//     tile against the same activation tile, B items two k-blocks;
//     every pair is one M = 128 x N = (tokens rounded up to 16) x K = 128
//     product, four MMAs of K = 32, into its own tensor-memory accumulator;
//   * the block scales are fp32 per 128 x 128 weight block and per token per
//     128 activation columns, so they cannot ride in the MMA: the epilogue
//     reads each k-block's partial product with tcgen05.ld (one row per
//     thread), multiplies it by (weight scale x token scale) and accumulates
//     in registers; at the end of a pass an A item applies the SwiGLU and
//     quantises h in registers (the group's amax is combined over the four
//     lane-quadrant warps through shared memory), a B item stores its rows.
// Routed tokens' activation rows come pre-gathered in route order (the
// gather kernel below), so that every activation tile is a contiguous TMA
// box.  Every wait is bounded (~0.2 s) and on expiry records
// MOE_ERR_DEVICE_TIMEOUT; the MMA warp waits for its own MMAs and the
// producer for its own copies before the CTA frees its tensor memory and
// ends.
#include <cuda.h>

#include <algorithm>

#include "async.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tmap.h"
#include "../../include/moe_decode.h"

namespace moe {

namespace {

constexpr int kRows = 128;               // weight rows of a tile: the MMA's M
constexpr int kPass = 64;                // tokens of a pass at most: the MMA's N
constexpr int kWTile = kRows * 128;      // one weight tile (128 rows x one k-block), 16 KB
constexpr int kXTile = kPass * 128;      // one activation tile (64 rows x one k-block), 8 KB
constexpr int kSlotB = 2 * kWTile + 2 * kXTile;  // a stage: two weight and two activation tiles, 48 KB
constexpr int kNST = 4;                  // ring stages
constexpr int kTCols = 512;              // tensor-memory columns: kNST accumulator pairs of 2 x kPass
constexpr int kMetaInts = 8;
constexpr int kThreads = 12 * 32;
constexpr int kPW = 0, kMW = 1, kSW = 2, kEW0 = 4, kNEpi = 8;
// Tuning constants of a dense layer's item split (measured on the DeepSeek-V3
// dense MLP; overridable at build time for sweeps).
#ifndef MOE_TC_W2_SEG_WAVES
#define MOE_TC_W2_SEG_WAVES 3
#endif
#ifndef MOE_TC_W13_SEGS
#define MOE_TC_W13_SEGS 1
#endif
constexpr int kSegWaves = MOE_TC_W2_SEG_WAVES;  // w2 items per SM, when a dense layer's I is split
constexpr int kW13Segs = MOE_TC_W13_SEGS; // K segments of a dense layer's w13 items

static_assert(kNST * 2 * kPass == kTCols, "one accumulator pair per ring stage");

// Shared-memory carve-up (byte offsets from the 1024-byte aligned base), used
// by the kernel and by the launch's size alike.
constexpr size_t align_to(size_t x, size_t a) { return (x + a - 1) / a * a; }
struct SmemTc {
  static constexpr size_t kMeta = (size_t)kNST * kSlotB;                        // stage descriptors
  static constexpr size_t kTmeta = kMeta + (size_t)kNST * kMetaInts * 4;        // accumulator descriptors
  static constexpr size_t kBars = kTmeta + (size_t)kNST * kMetaInts * 4;        // mbarriers
  static constexpr int kNBars = 6 * kNST + 4 + 3;
  static constexpr size_t kCstage = align_to(kBars + (size_t)kNBars * 8, 16);   // scale products (float4 reads)
  static constexpr size_t kAmax = kCstage + (size_t)kNST * 2 * kPass * 4;       // amax exchange
  static constexpr size_t kMisc = kAmax + 2 * 2 * 4 * 32 * 4;                    // misc words, then the tables
  static constexpr size_t bytes(int E) { return 1024 + kMisc + (size_t)(4 + 2 * E + 1) * 4; }
};
static_assert(SmemTc::kMeta % 1024 == 0 && SmemTc::kMeta % 16 == 0, "ring tiles 1024-aligned, descriptors 16");
static_assert(SmemTc::kTmeta % 16 == 0 && SmemTc::kBars % 8 == 0, "descriptor and barrier alignment");
static_assert(SmemTc::kCstage % 16 == 0 && SmemTc::kAmax % 16 == 0, "vector-read alignment");

// stage flags
enum TcFlag { kFA = 1, kFFirst = 2, kFLast = 4, kFEnd = 8, kFFinal = 16 };

// ------------------------------------------------------------- tcgen05 wrappers
// Shared-memory matrix descriptor of a K-major tile in the 128-byte swizzled
// layout TMA writes: 8-row atoms of 1024 bytes (stride-dimension offset), the
// leading-dimension offset unused, descriptor version 1, swizzle mode 2.
MOE_DEV uint64_t smem_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f8f6f4: fp32 accumulator, A and B E4M3,
// both K-major, N = n, M = 128.
MOE_DEV uint32_t instr_desc(int n) { return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24); }
MOE_DEV void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, int accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// the mbarrier receives one arrival once every MMA this thread issued so far is complete
MOE_DEV void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
               : "memory");
}
MOE_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MOE_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 16 consecutive fp32 columns of this thread's lane, without waiting: the
// registers are valid after tc_wait_ld()
MOE_DEV void tc_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}
MOE_DEV void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Bounded wait that ignores the status word (the waits of the MMA and
// epilogue warps end together, by the phase or by the bound).
MOE_DEV bool mbar_wait_t(uint64_t* b, uint32_t parity, int* status) { return mbar_wait_landed(b, parity, status); }

// ------------------------------------------------------------- work items
struct TcArgs {
  const uint8_t* xg;
  int sh_segs;     // K segments of the shared slot's w2 items (partial rows the boundary adds)
  int a_segs;      // K segments of the shared slot's w13 items (partial [g; u] rows in gu_part)
  float* gu_part;  // [group][segment][gate | up][kPass columns][128 rows] fp32
  int* pcount;     // [group] segments of the group done
};

struct TcItem {
  bool a;
  int slot, idx, seg;  // idx: 128-intermediate block (A) or 128-row block of w2 (B); seg: K segment (B)
};

struct TcSlot {
  int Ie;     // intermediate size of the expert
  int nt;     // tokens
  int o;      // first position in the route order (routed)
  int hbase;  // first h row
  int e;      // routed expert id, -1 for the shared expert
};

// A items: the shared slot's (128-intermediate block, K segment) pairs, then
// each routed expert's blocks; B items: the shared slot's (128-row block, K
// segment) pairs, then each routed expert's row blocks.
MOE_DEV TcItem tc_decode(int item, int nA_sh, int nA_r, int totA, int nB, const TcArgs& q, bool has_shared) {
  TcItem it;
  if (item < totA) {
    it.a = true;
    if (item < nA_sh) {
      it.slot = 0;
      it.idx = item / q.a_segs;
      it.seg = item % q.a_segs;
    } else {
      const int j = item - nA_sh;
      it.slot = j / nA_r + (has_shared ? 1 : 0);
      it.idx = j % nA_r;
      it.seg = 0;
    }
  } else {
    it.a = false;
    int j = item - totA;
    const int nBs = has_shared ? nB * q.sh_segs : 0;
    if (j < nBs) {
      it.slot = 0;
      it.idx = j / q.sh_segs;
      it.seg = j % q.sh_segs;
    } else {
      j -= nBs;
      it.slot = j / nB + (has_shared ? 1 : 0);
      it.idx = j % nB;
      it.seg = 0;
    }
  }
  return it;
}

MOE_DEV TcSlot tc_slot(const ExpertArgs& p, const int* s_off, const int* s_act, int slot, bool has_shared) {
  TcSlot s;
  if (has_shared && slot == 0) {
    s.Ie = p.Is; s.nt = p.M; s.o = 0; s.hbase = p.Mk; s.e = -1;
  } else {
    s.e = s_act[slot - (has_shared ? 1 : 0)];
    s.Ie = p.I; s.o = s_off[s.e]; s.nt = s_off[s.e + 1] - s.o; s.hbase = s.o;
  }
  return s;
}

// K range of an item, in k-blocks: segment seg of H (A) or of Ie (B)
MOE_DEV void tc_krange(const ExpertArgs& p, const TcItem& it, const TcSlot& s, const TcArgs& q, int& k0, int& k1) {
  const int nkb = it.a ? p.H / kBlock : s.Ie / kBlock;
  const int segs = s.e < 0 ? (it.a ? q.a_segs : q.sh_segs) : 1;
  // balanced: every segment holds at least one k-block (segs <= nkb)
  k0 = it.seg * nkb / segs;
  k1 = (it.seg + 1) * nkb / segs;
}

struct TcMaps {
  CUtensorMap w13, w2, sw13, sw2;  // weights, box 128 B x 128 rows
  CUtensorMap xq;                  // x codes [M][H], box 128 B x 16 rows
  CUtensorMap xg;                  // routed x codes gathered in route order [Mk][H]
  CUtensorMap hq;                  // h codes [Mk + M][Imax]
};


__global__ void __launch_bounds__(kThreads, 1)
    experts_tc_kernel(ExpertArgs p, TcArgs q, const __grid_constant__ TcMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (su32(smem_raw) & 1023)) & 1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nkbH = p.H / kBlock;

  // ---- shared memory (offsets in SmemTc): ring | stage descriptors | accumulator descriptors |
  //      barriers | scale products | amax exchange | tables
  uint8_t* ring = smem;
  int* meta = reinterpret_cast<int*>(smem + SmemTc::kMeta);      // [kNST][kMetaInts]
  int* tmeta = reinterpret_cast<int*>(smem + SmemTc::kTmeta);    // [kNST][kMetaInts]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SmemTc::kBars);
  uint64_t* empty = full + kNST;
  uint64_t* tfull = empty + kNST;
  uint64_t* tempty = tfull + kNST;
  uint64_t* mready = tempty + kNST;     // the producer has described the stage
  uint64_t* sready = mready + kNST;     // the stage's scale products are in cstage
  uint64_t* amax_bar = sready + kNST;   // [2 alternating buffers][2 column halves]
  uint64_t* mma_done = amax_bar + 4;
  uint64_t* psync = mma_done + 1;       // split w13 items: the eight warps wrote their partial sums
  uint64_t* pdec = psync + 1;           // split w13 items: whether this item completes its group
  float* cstage = reinterpret_cast<float*>(smem + SmemTc::kCstage);    // [kNST][2 pairs][kPass columns]
  float* amax_buf = reinterpret_cast<float*>(smem + SmemTc::kAmax);    // [2][2][4][32]
  int* s_misc = reinterpret_cast<int*>(smem + SmemTc::kMisc);          // [0] tensor-memory base, [1] routed experts, [2] split decision
  int* s_off = s_misc + 4;                                               // [E+1]
  int* s_act = s_off + (p.E + 1);                                        // [E]
  int* status = p.hdr + kHdrStatus;

  // the dynamic shared memory must start where the carve-up expects (checked
  // once; the condition is the same in every thread, so all leave together)
  if ((su32(ring) & 1023u) != 0) {
    if (tid == 0) atomicExch(status, MOE_ERR_INVALID_ARG);
    return;
  }
  if (tid == 0) {
    for (int i = 0; i < kNST; ++i) {
      mbar_init(full + i, 1);    // the producer's expect-tx arrival
      mbar_init(empty + i, 3);   // the MMAs' commit, the MMA thread, the scale warp (descriptor read)
      mbar_init(tfull + i, 2);   // the MMAs' commit + the MMA thread
      mbar_init(tempty + i, kNEpi);
      mbar_init(mready + i, 1);
      mbar_init(sready + i, 1);
    }
    for (int i = 0; i < 4; ++i) mbar_init(amax_bar + i, 4);
    mbar_init(mma_done, 1);
    mbar_init(psync, kNEpi);
    mbar_init(pdec, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_misc[1] = 0;
  }
  if (warp == kMW) {
    // the whole tensor memory of the SM (one CTA per SM)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(s_misc)),
                 "r"(kTCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  grid_dep_launch();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = (uint32_t)s_misc[0];

  const bool has_shared = p.Is > 0;
  const int nA_sh = has_shared ? p.Is / kRows * q.a_segs : 0;
  const int nA_r = p.I / kRows;
  const int nB = p.H / kRows;

  if (warp == kPW) {
    // ================================================================ producer
    uint32_t gs = 0;   // stages issued
    int si = 0;
    uint32_t ph = 0;
    bool alive = true, routed = false, all_ready = false;
    int totA = nA_sh, total = nA_sh;
    int item = 0;
    if (lane == 0) {
      // the router's first phase: x codes written, counters reset
      const unsigned long long t0 = globaltimer_ns();
      for (long n = 0;; ++n) {
        if (ld_acquire(p.hdr + kHdrXReady) >= p.router_ctas) break;
        if (*(volatile int*)status != 0 || n > (1l << 24)) { alive = false; break; }
        if (globaltimer_ns() - t0 > kWaitNs) {
          atomicExch(status, MOE_ERR_DEVICE_TIMEOUT);
          alive = false;
          break;
        }
        __nanosleep(64);
      }
      asm volatile("fence.proxy.async.global;" ::: "memory");  // x codes are read with TMA
      if (alive) item = atomicAdd(p.hdr + kHdrQueue, 1);
    }
    alive = __shfl_sync(0xffffffffu, alive, 0);
    item = __shfl_sync(0xffffffffu, item, 0);
    if (p.E == 0) {  // a dense layer: no routing to wait for
      routed = true;
      total = totA + nB * q.sh_segs;
    }
    while (alive) {
      if (item >= nA_sh && !routed) {
        // every routed item needs the routing (and the gathered rows): the
        // grids before this one are complete and their writes visible
        grid_dep_wait();
        asm volatile("fence.proxy.async.global;" ::: "memory");  // gathered rows are read with TMA
        int n_act = 0;
        if (lane == 0) n_act = __ldcg(p.hdr + kHdrActive);
        for (int i = lane; i <= p.E; i += 32) s_off[i] = __ldcg(p.off + i);
        for (int i = lane; i < min(p.E, p.Mk); i += 32) s_act[i] = __ldcg(p.act + i);
        n_act = __shfl_sync(0xffffffffu, n_act, 0);
        if (lane == 0) s_misc[1] = n_act;
        __syncwarp();
        totA = nA_sh + n_act * nA_r;
        total = totA + (has_shared ? nB * q.sh_segs : 0) + n_act * nB;
        routed = true;
      }
      if (item >= total) break;
      // the next item is claimed two stages before this one's last stage, not
      // now: with few, long items a claim made at the start would hold an item
      // that an idle CTA could run at once
      int nxt = 0;
      bool claimed = false;
      const TcItem it = tc_decode(item, nA_sh, nA_r, totA, nB, q, has_shared);
      const TcSlot s = tc_slot(p, s_off, s_act, it.slot, has_shared);
      int k0, k1;
      tc_krange(p, it, s, q, k0, k1);
      if (!it.a && !all_ready) {
        // a w2 item needs its K range of h quantised: every A item done, or
        // each group of the range published by all eight epilogue warps
        int ok = 0;
        if (lane == 0) ok = ld_acquire(p.hdr + kHdrDoneA) >= totA;
        if (__shfl_sync(0xffffffffu, ok, 0)) {
          all_ready = true;
        } else {
          const unsigned long long t0 = globaltimer_ns();
          for (int g0 = k0; g0 < k1 && alive; g0 += 32) {
            const int g = g0 + lane;
            for (long n = 0;; ++n) {
              const bool mine = g >= k1 || ld_acquire(p.gcount + it.slot * p.gI + g) >= kNEpi;
              if (__all_sync(0xffffffffu, mine)) break;
              int stop = 0;  // decided by lane 0 alone, so that the warp leaves together
              if (lane == 0) {
                if (*(volatile int*)status != 0 || n > (1l << 24)) {
                  stop = 1;
                } else if (globaltimer_ns() - t0 > kWaitNs) {
                  atomicExch(status, MOE_ERR_DEVICE_TIMEOUT);
                  stop = 1;
                }
              }
              if (__shfl_sync(0xffffffffu, stop, 0)) { alive = false; break; }
              __nanosleep(64);
            }
          }
          if (!alive) break;
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");  // h codes are read with TMA
      }
      const int passes = (s.nt + kPass - 1) / kPass;
      const int kstep = it.a ? 1 : 2;
      const int nstages = passes * ((k1 - k0 + kstep - 1) / kstep);
      int stage = 0;
      for (int pass = 0; pass < passes && alive; ++pass) {
        const int ntok = min(kPass, s.nt - pass * kPass);
        const int npad = (ntok + 15) & ~15;
        // activation rows of the pass: x rows (shared expert, dense), gathered
        // x rows in route order (routed), h rows (w2)
        const CUtensorMap* xmap = it.a ? (s.e < 0 ? &maps.xq : &maps.xg) : &maps.hq;
        const int xrow = (it.a ? (s.e < 0 ? 0 : s.o) : s.hbase) + pass * kPass;
        for (int kb = k0; kb < k1; kb += kstep, ++stage) {
          if (!claimed && stage >= nstages - 3) {
            if (lane == 0) nxt = atomicAdd(p.hdr + kHdrQueue, 1);
            claimed = true;
          }
          int ok = 1;
          if (lane == 0) ok = mbar_wait(empty + si, ph ^ 1u, status);
          __syncwarp();
          if (!__shfl_sync(0xffffffffu, ok, 0)) { alive = false; break; }
          const int nkv = min(kstep, k1 - kb);
          uint8_t* st = ring + (size_t)si * kSlotB;
          if (lane == 0) {
            int* md = meta + kMetaInts * si;
            const int fl = (it.a ? kFA : 0) | (kb == k0 ? kFFirst : 0) | (kb + kstep >= k1 ? kFLast : 0) |
                           (kb + kstep >= k1 && pass == passes - 1 ? kFFinal : 0);
            *reinterpret_cast<int4*>(md) = make_int4(item, pass, kb, fl);
            *reinterpret_cast<int4*>(md + 4) = make_int4(ntok, npad, nkv, 0);
            mbar_arrive(mready + si);  // the scale warp starts on the descriptor now
            const uint32_t xbytes = (uint32_t)(npad / 16) * 2048u;
            mbar_expect_tx(full + si, it.a ? 2u * kWTile + xbytes : (uint32_t)nkv * (kWTile + xbytes));
          }
          __syncwarp();
          // one copy per lane: lanes 0/1 the weight tiles (A: gate, up; B: k-blocks
          // kb, kb + 1), lanes 2.. the 16-row activation boxes of each k-block
          const int nxb = npad / 16;
          if (lane < 2) {
            if (it.a) {
              const int row = (s.e < 0 ? 0 : s.e * 2 * s.Ie) + lane * s.Ie + kRows * it.idx;
              tma_load_2d(st + lane * kWTile, s.e < 0 ? &maps.sw13 : &maps.w13, kb * kBlock, row, full + si);
            } else if (lane < nkv) {
              const int row = (s.e < 0 ? 0 : s.e * p.H) + kRows * it.idx;
              tma_load_2d(st + lane * kWTile, s.e < 0 ? &maps.sw2 : &maps.w2, (kb + lane) * kBlock, row, full + si);
            }
          } else {
            const int c = lane - 2, j = c / nxb, b = c % nxb;  // k-block j of the stage, box b
            if (c < (it.a ? 1 : nkv) * nxb)
              tma_load_2d(st + 2 * kWTile + j * kXTile + b * 2048, xmap, (kb + j) * kBlock, xrow + 16 * b, full + si);
          }
          ++gs;
          if (++si == kNST) { si = 0; ph ^= 1u; }
        }
        __syncwarp();
      }
      if (!claimed && lane == 0) nxt = atomicAdd(p.hdr + kHdrQueue, 1);  // (an item that stopped early)
      item = __shfl_sync(0xffffffffu, nxt, 0);
    }
    // end marker, then make sure every copy this CTA issued has landed
    {
      int ok = 1;
      if (lane == 0) ok = mbar_wait_landed(empty + si, ph ^ 1u, status);
      if (__shfl_sync(0xffffffffu, ok, 0)) {
        if (lane == 0) {
          meta[kMetaInts * si + 3] = kFEnd;
          mbar_arrive(mready + si);
          mbar_arrive(full + si);
        }
        ++gs;
      }
    }
    if (lane == 0)
      for (uint32_t j = (gs > (uint32_t)kNST ? gs - kNST : 0); j < gs; ++j)
        mbar_wait_landed(full + (j % kNST), (j / kNST) & 1u, status);
    __syncwarp();
  } else if (warp == kMW) {
    // ================================================================ MMA issue
    if (lane == 0) {
      int si = 0;
      uint32_t ph = 0;
      bool issued = false;
      while (true) {
        if (!mbar_wait_t(full + si, ph, status)) break;
        const int* md = meta + kMetaInts * si;
        const int4 m0 = *reinterpret_cast<const int4*>(md);
        const int4 m1 = *reinterpret_cast<const int4*>(md + 4);
        // the accumulator pair of this stage: free once the epilogue has read it
        if (!mbar_wait_t(tempty + si, ph ^ 1u, status)) break;
        int* tm = tmeta + kMetaInts * si;
        *reinterpret_cast<int4*>(tm) = m0;
        *reinterpret_cast<int4*>(tm + 4) = m1;
        if (m0.w & kFEnd) {
          mbar_arrive(tfull + si);
          mbar_arrive(tfull + si);
          break;
        }
        tc_fence_after();
        const bool a = (m0.w & kFA) != 0;
        const int npad = m1.y, nkv = m1.z;
        const uint32_t idesc = instr_desc(npad);
        const uint32_t sb = su32(ring + (size_t)si * kSlotB);
        for (int pr = 0; pr < 2; ++pr) {
          if (!a && pr >= nkv) break;
          const uint64_t da = smem_desc(sb + pr * kWTile);
          const uint64_t db = smem_desc(sb + 2 * kWTile + (a ? 0 : pr) * kXTile);
          const uint32_t dt = tmem + (uint32_t)(si * 2 * kPass + pr * kPass);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) tc_mma(dt, da + 2 * kk, db + 2 * kk, idesc, kk > 0 ? 1 : 0);
        }
        issued = true;
        tc_commit(tfull + si);   // the accumulators are complete
        mbar_arrive(tfull + si);
        tc_commit(empty + si);   // the stage's tiles are read
        mbar_arrive(empty + si);
        if (++si == kNST) { si = 0; ph ^= 1u; }
      }
      // every MMA this thread issued has completed before the memory is freed
      if (issued) {
        tc_commit(mma_done);
        mbar_wait_landed(mma_done, 0, status);
      }
    }
    __syncwarp();
  } else if (warp == kSW) {
    // ================================================================ scale products
    // For every stage, as soon as the producer has described it: the scale of
    // each (pair, token column): weight block scale x token group scale, so
    // that the epilogue reads them from shared memory.  x scales through L1;
    // h scales from L2 (a split w2 item may meet a 128-byte line of them
    // whose other groups another CTA writes later).
    int si = 0;
    uint32_t ph = 0;
    int cur_item = -1, cur_pass = -1;
    TcItem it{};
    TcSlot s{};
    const float* ws0 = nullptr;
    const float* ws1 = nullptr;
    const float* xsr[2] = {nullptr, nullptr};  // scale rows of this lane's columns lane, lane + 32
    while (true) {
      if (!mbar_wait_t(mready + si, ph, status)) break;
      const int* md = meta + kMetaInts * si;
      const int4 m0 = *reinterpret_cast<const int4*>(md);
      const int4 m1 = *reinterpret_cast<const int4*>(md + 4);
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + si);  // the descriptor is read
      if (m0.w & kFEnd) break;
      const int item = m0.x, pass = m0.y, kb = m0.z, ntok = m1.x, nkv = m1.z;
      const bool a = (m0.w & kFA) != 0;
      if (item != cur_item) {
        cur_item = item;
        cur_pass = -1;
        const int n_act = *(volatile int*)(s_misc + 1);
        it = tc_decode(item, nA_sh, nA_r, nA_sh + n_act * nA_r, nB, q, has_shared);
        s = tc_slot(p, s_off, s_act, it.slot, has_shared);
        if (it.a) {
          const float* base = s.e < 0 ? p.sw13_s : p.w13_s + (size_t)s.e * (2 * p.I / kBlock) * nkbH;
          ws0 = base + (size_t)it.idx * nkbH;
          ws1 = base + (size_t)(s.Ie / kBlock + it.idx) * nkbH;
        } else {
          const int nkbI = s.Ie / kBlock;
          ws0 = (s.e < 0 ? p.sw2_s : p.w2_s + (size_t)s.e * nkbH * (p.I / kBlock)) + (size_t)it.idx * nkbI;
          ws1 = ws0;
        }
      }
      if (pass != cur_pass) {
        cur_pass = pass;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = lane + 32 * h, tl = pass * kPass + c;
          xsr[h] = nullptr;
          if (c < ntok) {
            if (a) {
              const int tok = s.e < 0 ? tl : __ldcg(p.sorted + s.o + tl) / p.k;
              xsr[h] = p.xs + (size_t)tok * nkbH;
            } else {
              xsr[h] = p.hs + (size_t)(s.hbase + tl) * p.hsS;
            }
          }
        }
      }
      // the previous use of this stage's products has been read by the epilogue
      if (!mbar_wait_t(tempty + si, ph ^ 1u, status)) break;
      float* cs = cstage + si * 2 * kPass;
      const float w0 = ld_ca(ws0 + kb);
      const float w1 = a ? ld_ca(ws1 + kb) : (nkv > 1 ? ld_ca(ws0 + kb + 1) : 0.f);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = lane + 32 * h;
        float c0 = 0.f, c1 = 0.f;
        if (xsr[h]) {
          if (a) {
            const float sx = ld_ca(xsr[h] + kb);
            c0 = w0 * sx;
            c1 = w1 * sx;
          } else {
            c0 = w0 * __ldcg(xsr[h] + kb);
            c1 = nkv > 1 ? w1 * __ldcg(xsr[h] + kb + 1) : 0.f;
          }
        }
        cs[c] = c0;
        cs[kPass + c] = c1;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(sready + si);
      if (++si == kNST) { si = 0; ph ^= 1u; }
    }
  } else if (warp >= kEW0) {
    // ================================================================ epilogue
    // Warp (qd, hf) owns rows 32 qd .. 32 qd + 31 of the 128-row tile and the
    // 16-column blocks hf and 2 + hf of a pass: accumulator index j < 16 is
    // column 16 hf + j, j >= 16 column 32 + 16 hf + (j - 16), so that passes
    // of up to 32 tokens still keep all eight warps busy.
    const int ew = warp - kEW0;
    const int qd = warp & 3;           // tensor-memory lane quadrant
    const int hf = ew >> 2;
    const int r = 32 * qd + lane;      // this thread's row of the 128-row tile
    const int colA = 16 * hf, colB = 32 + 16 * hf;
    const int my_col = lane < 16 ? colA + lane : colB + lane - 16;  // this lane's column (pass ends)
    float acc0[32], acc1[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) acc0[j] = acc1[j] = 0.f;
    int cur_item = -1;
    TcItem it{};
    TcSlot s{};
    uint32_t pe = 0;  // A-item pass ends so far: the amax buffer and barrier alternate with it
    uint32_t pu = 0;  // split w13 item ends so far (psync / pdec phases)
    int si = 0;
    uint32_t ph = 0;
    while (true) {
      if (!mbar_wait_t(tfull + si, ph, status)) break;
      const int* tm = tmeta + kMetaInts * si;
      const int4 m0 = *reinterpret_cast<const int4*>(tm);
      const int4 m1 = *reinterpret_cast<const int4*>(tm + 4);
      if (m0.w & kFEnd) break;
      const int item = m0.x, pass = m0.y, fl = m0.w, ntok = m1.x, nkv = m1.z;
      const bool a = (fl & kFA) != 0;
      if (!mbar_wait_t(sready + si, ph, status)) break;
      tc_fence_after();
      const bool blkA = colA < ntok, blkB = colB < ntok;  // (warp-uniform) blocks holding tokens
      const bool two = a || nkv > 1;                      // the stage's second accumulator is live
      if (blkA || blkB) {
        const uint32_t ta = tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(si * 2 * kPass);
        const float* cs = cstage + si * 2 * kPass;
        float d[32];
        // the first accumulator of the stage (gate rows, or the first k-block)
        if (blkA) tc_ld16(ta + colA, d);
        if (blkB) tc_ld16(ta + colB, d + 16);
        tc_wait_ld();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (h == 0 ? !blkA : !blkB) continue;
          const int col = h == 0 ? colA : colB;
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            const float4 f0 = *reinterpret_cast<const float4*>(cs + col + j);
            const int i = 16 * h + j;
            acc0[i] += d[i] * f0.x; acc0[i + 1] += d[i + 1] * f0.y;
            acc0[i + 2] += d[i + 2] * f0.z; acc0[i + 3] += d[i + 3] * f0.w;
          }
        }
        if (two) {
          // the second: up rows (A) or the stage's second k-block (B)
          if (blkA) tc_ld16(ta + kPass + colA, d);
          if (blkB) tc_ld16(ta + kPass + colB, d + 16);
          tc_wait_ld();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (h == 0 ? !blkA : !blkB) continue;
            const int col = h == 0 ? colA : colB;
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
              const float4 f1 = *reinterpret_cast<const float4*>(cs + kPass + col + j);
              const int i = 16 * h + j;
              if (a) {
                acc1[i] += d[i] * f1.x; acc1[i + 1] += d[i + 1] * f1.y;
                acc1[i + 2] += d[i + 2] * f1.z; acc1[i + 3] += d[i + 3] * f1.w;
              } else {
                acc0[i] += d[i] * f1.x; acc0[i + 1] += d[i + 1] * f1.y;
                acc0[i + 2] += d[i + 2] * f1.z; acc0[i + 3] += d[i + 3] * f1.w;
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty + si);
      if (++si == kNST) { si = 0; ph ^= 1u; }
      if (!(fl & kFLast)) continue;

      // ---- end of a pass
      if (item != cur_item) {
        cur_item = item;
        const int n_act = *(volatile int*)(s_misc + 1);
        it = tc_decode(item, nA_sh, nA_r, nA_sh + n_act * nA_r, nB, q, has_shared);
        s = tc_slot(p, s_off, s_act, it.slot, has_shared);
      }
      const int tl_me = pass * kPass + my_col;  // this lane's token of the slot (if my_col < ntok)
      const int nA = min(16, max(0, ntok - colA)), nB = min(16, max(0, ntok - colB));  // tokens in each block
      if (!a) {
        // w2: this thread's row of every token's output (fp32), unweighted
        const int hrow = kRows * it.idx + r;
        float* base = s.e < 0 ? p.shared_out + (size_t)it.seg * p.M * p.H : p.rows;
        const int out_row = my_col < ntok ? (s.e < 0 ? tl_me : __ldcg(p.sorted + s.o + tl_me)) : 0;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (j < 16 ? j < nA : j - 16 < nB) {
            const int orow = __shfl_sync(0xffffffffu, out_row, j);
            base[(size_t)orow * p.H + hrow] = acc0[j];
          }
        }
      } else {
        const int grp = it.idx;  // the item's 128 intermediates are h group idx
        if (s.e < 0 && q.a_segs > 1) {
          // a K segment of a split w13 item: its partial [g; u] rows go to the
          // workspace; the item that completes the group adds every segment's
          // rows in segment order and goes on below, the others are done
          const size_t gbase = (size_t)grp * q.a_segs * 2 * kPass * kRows;
          float* part = q.gu_part + gbase + (size_t)it.seg * 2 * kPass * kRows;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = j < 16 ? colA + j : colB + j - 16;
            if (col < ntok) {
              part[(size_t)col * kRows + r] = acc0[j];
              part[(size_t)(kPass + col) * kRows + r] = acc1[j];
            }
          }
          __threadfence();
          __syncwarp();
          if (lane == 0) mbar_arrive(psync);
          if (!mbar_wait_t(psync, pu & 1u, status)) break;
          if (ew == 0 && lane == 0) {
            __threadfence();
            const int last = atomicAdd(q.pcount + grp, 1) == q.a_segs - 1;
            s_misc[2] = last;
            if (!last) atomicAdd(p.hdr + kHdrDoneA, 1);  // (the completing item counts when it publishes)
            mbar_arrive(pdec);
          }
          const bool ok = mbar_wait_t(pdec, pu & 1u, status);
          ++pu;
          if (!ok) break;
          if (!*(volatile int*)(s_misc + 2)) {
#pragma unroll
            for (int j = 0; j < 32; ++j) acc0[j] = acc1[j] = 0.f;
            continue;
          }
          __threadfence();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = j < 16 ? colA + j : colB + j - 16;
            float g = 0.f, u = 0.f;
            if (col < ntok)
              for (int sg = 0; sg < q.a_segs; ++sg) {
                const float* ps = q.gu_part + gbase + (size_t)sg * 2 * kPass * kRows;
                g += __ldcg(ps + (size_t)col * kRows + r);
                u += __ldcg(ps + (size_t)(kPass + col) * kRows + r);
              }
            acc0[j] = g;
            acc1[j] = u;
          }
        }
        // w13: h = silu(min(g, L)) * clamp(u, -L, L) for the columns that hold
        // tokens (the counts are the same in the whole warp), then FP8 per token
        // over the 128 intermediates of this item (the four lane quadrants of
        // the column half)
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (j < 16 ? j < nA : j - 16 < nB) {
            const float z = fminf(acc0[j], p.limit);
            acc0[j] = __fdividef(z, 1.f + __expf(-z)) * fminf(fmaxf(acc1[j], -p.limit), p.limit);
            acc1[j] = fabsf(acc0[j]);
          } else {
            acc1[j] = 0.f;
          }
        }
        // per-column max over this warp's 32 rows: after the five exchange
        // steps lane l holds the max of accumulator column l
#pragma unroll
        for (int sh = 16; sh >= 1; sh >>= 1) {
          const bool upper = (lane & sh) != 0;
#pragma unroll
          for (int i = 0; i < sh; ++i) {
            const float send = upper ? acc1[i] : acc1[i + sh];
            const float keep = upper ? acc1[i + sh] : acc1[i];
            acc1[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, sh));
          }
        }
        const int pb = pe & 1;
        float* ab = amax_buf + (pb * 2 + hf) * 4 * 32;
        ab[qd * 32 + lane] = acc1[0];
        __syncwarp();
        if (lane == 0) mbar_arrive(amax_bar + pb * 2 + hf);
        const bool ok = mbar_wait_t(amax_bar + pb * 2 + hf, (pe >> 1) & 1u, status);
        ++pe;
        if (!ok) break;
        const float amax = fmaxf(fmaxf(ab[lane], ab[32 + lane]), fmaxf(ab[64 + lane], ab[96 + lane]));
        const float scl = group_scale(amax, p.e8m0 != 0);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (j < 16 ? j < nA : j - 16 < nB) {
            const int col = j < 16 ? colA + j : colB + j - 16;
            const float sj = __shfl_sync(0xffffffffu, scl, j);
            const size_t row = (size_t)(s.hbase + pass * kPass + col);
            uint16_t code;
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(code) : "f"(0.f), "f"(__fdiv_rn(acc0[j], sj)));
            p.hq[row * p.Imax + grp * kBlock + r] = (uint8_t)(code & 0xff);
          }
        }
        if (qd == 0 && my_col < ntok) p.hs[(size_t)(s.hbase + tl_me) * p.hsS + grp] = scl;
        if (fl & kFFinal) {
          // this warp's part of the group is written: publish it (the codes are
          // read with TMA by other CTAs); the eighth warp counts the item
          asm volatile("fence.proxy.async.global;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            __threadfence();
            const bool withhold = p.hdr[kHdrFault] != 0 && it.slot == 0;
            if (!withhold && atomicAdd(p.gcount + it.slot * p.gI + grp, 1) == kNEpi - 1) {
              __threadfence();
              atomicAdd(p.hdr + kHdrDoneA, 1);
            }
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) acc0[j] = acc1[j] = 0.f;
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == kMW) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTCols) : "memory");
  }
  if (tid == 0) {
    // the last CTA to finish clears the router's x-ready count for the next call
    __threadfence();
    if (atomicAdd(p.hdr + kHdrExit, 1) == (int)gridDim.x - 1) {
      p.hdr[kHdrXReady] = 0;
      p.hdr[kHdrExit] = 0;
    }
  }
}

// Routed tokens' x codes copied into route order (row p = x row of the
// token of route sorted[p]), so that the tensor-core kernel reads each
// expert's tokens as one contiguous tile.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint8_t* xq, const int* sorted, int k, int Mk, int H,
                                                          uint8_t* xg) {
  grid_dep_launch();
  grid_dep_wait();  // the route order of the router kernel
  const int n16 = H / 16;
  for (int pr = blockIdx.x; pr < Mk; pr += gridDim.x) {
    const int t = __ldcg(sorted + pr) / k;
    const uint4* src = reinterpret_cast<const uint4*>(xq + (size_t)t * H);
    uint4* dst = reinterpret_cast<uint4*>(xg + (size_t)pr * H);
    for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = __ldcg(src + i);
  }
}

size_t tc_smem_bytes(int E) { return SmemTc::bytes(E); }

}  // namespace

int tc_w13_segments(int E, int H, int Is, int M) {
  // a dense layer's w13 items (one per 128 intermediates: fewer than a wave
  // of SMs can balance) are split four ways over H while one pass holds all
  // tokens, so that groups complete in several waves and the w2 items start
  // behind them; the completing segment adds the partial rows
  return (E == 0 && Is > 0 && M <= kPass) ? std::min(kW13Segs, H / kBlock) : 1;
}

size_t tc_w13_partial_bytes(int E, int Is) {
  return E == 0 && Is > 0 && kW13Segs > 1 ? (size_t)(Is / kBlock) * kW13Segs * 2 * kPass * kRows * sizeof(float) : 0;
}

int tc_shared_segments(int E, int H, int Is, int M, int num_sms) {
  // a dense layer's long w2 rows (I_s / 128 k-blocks) are split into K
  // segments while one pass holds all tokens: as many as make about three
  // equal items per SM (the w2 phase runs as whole waves), at most one per
  // k-block; the boundary adds the partial rows.  An MoE layer's shared
  // expert is one of many experts and is never split.
  if (E != 0 || Is <= 0 || M > kPass) return 1;
  const int nB = H / kRows;
  return std::max(1, std::min({Is / kBlock, kMaxSharedSegs, (kSegWaves * num_sms + nB / 2) / nB}));
}

static_assert(sizeof(TcMaps) <= sizeof(ExpertsLaunch::maps), "tensor maps fit the prepared launch");

cudaError_t prepare_experts_tc(const ExpertArgs& a, const TcExtra& x, ExpertsLaunch& L) {
  if (!encode_fn()) return cudaErrorNotSupported;
  memset(&L, 0, sizeof(L));
  L.a = a;
  L.tc = true;
  L.tcx = x;
  const uint8_t* xg = x.xg;
  TcMaps* maps = reinterpret_cast<TcMaps*>(L.maps);
  // weights: [rows][K] bytes, box one k-block x 128 rows; activations box one k-block x 16 rows
  if (a.E > 0 && (!tmap_2d(&maps->w13, a.w13, a.H, (uint64_t)a.E * 2 * a.I, 128, kRows) ||
                  !tmap_2d(&maps->w2, a.w2, a.I, (uint64_t)a.E * a.H, 128, kRows) ||
                  !tmap_2d(&maps->xg, xg, a.H, a.Mk, 128, 16)))
    return cudaErrorInvalidValue;
  if (a.Is > 0 && (!tmap_2d(&maps->sw13, a.sw13, a.H, 2 * (uint64_t)a.Is, 128, kRows) ||
                   !tmap_2d(&maps->sw2, a.sw2, a.Is, a.H, 128, kRows)))
    return cudaErrorInvalidValue;
  if (!tmap_2d(&maps->xq, a.xq, a.H, a.M, 128, 16) ||
      !tmap_2d(&maps->hq, a.hq, a.Imax, (uint64_t)a.Mk + a.M, 128, 16))
    return cudaErrorInvalidValue;
  L.smem = tc_smem_bytes(a.E);
  if (L.smem > 227 * 1024) return cudaErrorInvalidConfiguration;
  return cudaFuncSetAttribute(experts_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.smem);
}

cudaError_t launch_experts_tc_prepared(const ExpertsLaunch& L, int num_sms, cudaStream_t s) {
  TcMaps maps;
  memcpy(&maps, L.maps, sizeof(maps));
  TcArgs q;
  q.xg = L.tcx.xg;
  q.sh_segs = L.tcx.sh_segs;
  q.a_segs = L.tcx.a_segs;
  q.gu_part = L.tcx.gu_part;
  q.pcount = L.tcx.pcount;
  PdlLaunch P(dim3(num_sms), dim3(kThreads), L.smem, s);
  return cudaLaunchKernelEx(&P.cfg, experts_tc_kernel, L.a, q, maps);
}

cudaError_t launch_gather_rows(const uint8_t* xq, const int* sorted, int k, int Mk, int H, uint8_t* xg, int num_sms,
                               cudaStream_t s) {
  if (Mk <= 0) return cudaSuccess;
  PdlLaunch L(dim3(std::min(Mk, 2 * num_sms)), dim3(256), 0, s);
  return cudaLaunchKernelEx(&L.cfg, gather_rows_kernel, xq, sorted, k, Mk, H, xg);
}

}  // namespace moe
