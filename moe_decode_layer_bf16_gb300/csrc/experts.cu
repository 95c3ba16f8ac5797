// The routed + shared experts of one MoE decode step as one persistent kernel
// (the decode page, vllm.models.glm5next.nvidia.specialized_decode.runtime
// .decode, LayerStages._mega_moe: the routed experts in a single kernel; its
// grouped form folds the shared expert in as an extra expert, which this
// kernel does at every token count).
//
// Per expert: [g; u] = xq . w13^T with 128x128 block scales, clamped SwiGLU
// h = silu(min(g, L)) * clamp(u, -L, L), h re-quantised to FP8 per route per
// 128-column group, y = hq . w2^T.  Routed outputs are written unweighted, in
// expanded route order (the page's UnfinalizedMoEOutput rows with the
// identity expanded->permuted map); the shared expert's output separately.
//
// The step streams each active expert's FP8 weights exactly once and is
// HBM-bound at every token count of the workload, so the kernel is built as a
// weight stream that never drains:
//   * one CTA per SM: one producer warp, 16 consumer warps (8 when a pass
//     holds 16 tokens) and one epilogue warp, placed so that the producer
//     shares its sub-partition with little else;
//   * work items, taken by the producer from one atomic queue (all w13 items,
//     shared expert first, then all w2 items):
//       A item (expert, 16 intermediates): 16 gate + 16 up rows of w13 over H,
//       B item (expert, 128 rows of w2, one scale block) over I, streamed as
//       four 32-row groups (two per item when the whole-block items would be
//       too few to spread over the SMs, one when I is long: a dense MLP);
//   * a stage is 8 k-blocks (1024 columns): two 16 KB TMA boxes of weights
//     (128-byte swizzle) plus the pass's FP8 activation columns (TMA boxes of
//     the shared expert's x rows, or one 1-D bulk copy per token row), all
//     completing on the stage's mbarrier; the producer runs up to a whole
//     ring of stages ahead, across item boundaries, so epilogues overlap the
//     stream;
//   * each consumer warp takes one 16-row tile of one (or two) of the stage's
//     k-blocks (warp-level FP8 MMA, m16n8k32, fp32 accumulate, block scales
//     applied per k-block); the epilogue warp adds the k-block partial sums of
//     each 32-row group, handed over in shared memory.
// The A item that completes the 8th slice of a 128-column group quantises that
// group of h for every route; an expert's B items are issued once all of its
// groups are quantised.  Every wait is bounded (~0.2 s): on expiry the kernel
// records MOE_ERR_DEVICE_TIMEOUT in the workspace status word, skips the work
// and still ends, after its own copies in flight have landed.  Only items
// already taken by running CTAs are ever waited on, so the queue cannot
// deadlock however many CTAs are resident.
#include <cuda.h>

#include <algorithm>

#include "async.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tmap.h"
#include "../../include/moe_decode.h"

namespace moe {

namespace {

constexpr int kKBS = 8;                   // k-blocks per stage (two TMA boxes of 4)
constexpr int kKH = 4;                    // k-blocks per TMA box
constexpr int kSliceA = 16;               // intermediates per A item
constexpr int kRowsB = 128;               // w2 rows per B item (one scale block)
constexpr int kRowsQ = 32;                // w2 rows per stage (a quarter of a B item)
constexpr int kWBytes = 32768;            // weight tile per stage (two 16 KB boxes)
constexpr int kWHalf = 16384;
constexpr int kXStride = 1088;            // gathered activation row pitch in a stage (1024 + 64)
constexpr int kTabPer = 16;               // routing-table loads a producer lane keeps in flight
constexpr int kSmemMax = 227 * 1024;

// kFirst: first stage of a pass; kLast: last stage of a 32-row group (its
// epilogue runs); kPassEnd: last stage of the pass; kSkip: nothing was copied
// (the item gave up waiting), kEnd: no more work.  kXT: the stage's activation
// rows came as TMA boxes (swizzled), otherwise as one bulk copy per token
// (rows at a kXStride-byte pitch).  kA: a w13 item (x scales), else w2 (h scales).
enum MetaFlag { kFirst = 1, kLast = 2, kSkip = 4, kEnd = 8, kPassEnd = 16, kXT = 32, kA = 64 };

// Per ring slot, the producer describes the stage to the consumers so that they
// decode nothing themselves: ints [0, 4) item, pass | quarter << 16, first
// k-block, flags; [4] tokens of the pass, [5] valid k-blocks of the stage; at
// the first stage of a pass also [8, 12) the weight-scale rows of the two
// 16-row tiles (two pointers) and [16, 16 + tokens of the pass) each token's
// scale-row offset: Cfg<TT>::kMetaInts ints a slot.

template <int TT>
struct Cfg {
  static constexpr int kTok = 8 * TT;
  static constexpr int kXBytes = ((kTok * kXStride + 1023) / 1024) * 1024;
  static constexpr int kXHalf = kTok * kKH * 128;  // one activation box (tokens x 4 k-blocks)
  static constexpr int kSlot = kWBytes + kXBytes;
  // a stage descriptor: 16 ints, then one scale-row offset per token of the
  // pass (a multiple of 4 ints, for the 16-byte stores); as small as it can
  // be, since at 8-token passes the ring's fifth stage fits with little room
  static constexpr int kMetaInts = 16 + kTok;
  static_assert(kMetaInts % 4 == 0, "16-byte aligned descriptors");
  static_assert(TT == 1 || TT == 2 || TT == 4, "passes of 8, 16 or 32 tokens");
  static constexpr int kRedBufs = TT == 4 ? 1 : 2;  // epilogue hand-off buffers (one fits at 32 tokens)
  // consumer warps: each owns one 16-row tile and kKP of the stage's 8 k-blocks
  // (16 warps x 1 k-block where the registers allow, else 8 warps x 2)
  static constexpr int kCW = TT == 1 ? 16 : 8;
  static constexpr int kKP = 2 * kKBS / kCW;   // k-blocks per consumer warp and stage
  static constexpr int kKW = kKBS / kKP;       // k-block partial sums per tile
  // Warp roles.  An SM spreads a block's warps over its four sub-partitions by
  // warp index mod 4, and the producer warp, which issues every copy of the
  // stream, is the kernel's critical path: it gets sub-partition 0 with the
  // epilogue warp and at most one consumer (measured: 11% faster at 32 tokens
  // than sharing it with four consumers).  Warps 12 and 16 (8-token passes)
  // or 8 (16-token passes) only fill slots of that sub-partition and idle.
  static constexpr int kPW = 0;                // producer warp
  static constexpr int kEW = 4;                // epilogue warp
  static constexpr int kThreads = (TT == 1 ? 20 : 11) * 32;
  // consumer index of warp w (its rank among the consumer warps), -1 otherwise
  static __device__ __forceinline__ int consumer(int w) {
    if (TT == 1) return (w == 0 || w == 4 || w == 12 || w == 16) ? -1 : w - 1 - (w > 4) - (w > 12) - (w > 16);
    return (w % 4 == 0) ? -1 : w - 1 - (w > 4) - (w > 8);
  }
  static constexpr int kNSTMax = 5;
};

// ------------------------------------------------------------- work items
struct Slot {
  int Ie;      // intermediate size of this expert
  int nt;      // routes (tokens) of this expert
  int o;       // first position in the sorted route list (routed)
  int hbase;   // first h row
  int e;       // routed expert id (-1: shared)
};

struct Tables {
  const int* off;
  const int* act;
  const int* sorted;
};

struct Item {
  bool a;
  int slot, idx;  // slice (A) or 128-row block (B)
  int q0;         // B: first 32-row quarter of the block
};

// B items: bq quarters of a 128-row block each (4: the whole block)
MOE_DEV Item decode_item(int item, int nA_sh, int nA_r, int totA, int nB, bool has_shared, int bq) {
  Item it;
  if (item < totA) {
    it.a = true;
    if (item < nA_sh) { it.slot = 0; it.idx = item; }
    else { const int j = item - nA_sh; it.slot = j / nA_r + (has_shared ? 1 : 0); it.idx = j % nA_r; }
  } else {
    it.a = false;
    const int lp = bq == 4 ? 0 : bq == 2 ? 1 : 2;  // log2 of the items per 128-row block
    const int j = item - totA;
    it.slot = j / (nB << lp);
    const int r = j - it.slot * (nB << lp);
    it.idx = r >> lp;
    it.q0 = (r & ((1 << lp) - 1)) * bq;
  }
  return it;
}

MOE_DEV Slot make_slot(const ExpertArgs& p, const Tables& t, int slot, bool has_shared) {
  Slot s;
  if (has_shared && slot == 0) {
    s.Ie = p.Is; s.nt = p.M; s.o = 0; s.hbase = p.Mk; s.e = -1;
  } else {
    s.e = t.act[slot - (has_shared ? 1 : 0)];
    s.Ie = p.I; s.o = t.off[s.e]; s.nt = t.off[s.e + 1] - s.o; s.hbase = s.o;
  }
  return s;
}

MOE_DEV int token_of(const ExpertArgs& p, const Tables& t, const Slot& s, int i) {
  return s.e < 0 ? i : t.sorted[s.o + i] / p.k;
}

struct TmaMaps {
  CUtensorMap w13, w2, sw13, sw2;
  CUtensorMap xq;  // x codes [M][H/128][128], box 4 k-blocks x (tokens of a pass)
  CUtensorMap hq;  // h codes [Mk + M][Imax/128][128], same box
};

template <int TT>
__global__ void __launch_bounds__(Cfg<TT>::kThreads, 1) experts_kernel(ExpertArgs p, const __grid_constant__ TmaMaps maps,
                                                              int nst) {
  using C = Cfg<TT>;
  constexpr int kTok = C::kTok;
  constexpr int kCW = C::kCW, kKP = C::kKP, kKW = C::kKW, kPW = C::kPW, kEW = C::kEW, kThreads = C::kThreads;
  constexpr int kMetaInts = C::kMetaInts;
  constexpr int kRedF = 2 * kKW * 16 * kTok;  // floats of one epilogue hand-off buffer
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (su32(smem_raw) & 1023)) & 1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, q = lane & 3;
  const int nkbH = p.H / kBlock;

  // ---- shared memory carve-up: ring slots [W tile | activation rows | scales]
  uint8_t* ring = smem;
  int* meta = reinterpret_cast<int*>(smem + (size_t)nst * C::kSlot);              // [nst][kMetaInts]
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + kMetaInts * nst);            // [nst]
  uint64_t* empty = full + nst;                                                    // [nst]
  uint64_t* red_full = empty + nst;                                                // [2]
  uint64_t* red_empty = red_full + 2;                                              // [2]
  float* red = reinterpret_cast<float*>(red_empty + 2);                            // [bufs][2][kKW][16][kTok]
  int* epi = reinterpret_cast<int*>(red + C::kRedBufs * kRedF);                    // [2][4]
  int* s_off = epi + 8;                                                            // [E+1]
  int* s_act = s_off + (p.E + 1);                                                  // [E]
  int* s_sorted = s_act + p.E;                                                     // [Mk]
  int* s_misc = s_sorted + p.Mk;                                                   // [4]
  int* s_rdy = s_misc + 4;                                                         // [E+1]
  int* status = p.hdr + kHdrStatus;

  if (tid == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(full + i, 1);  // the producer's expect-tx arrival
      mbar_init(empty + i, kCW);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(red_full + b, kCW);
      mbar_init(red_empty + b, 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // The router kernel may still be running: the shared expert's w13 items need
  // only its first phase (x codes, counters reset), signalled by kHdrXReady;
  // the producer waits for the whole router grid (griddepcontrol.wait) before
  // its first routed item and then copies the routing tables to shared memory.
  grid_dep_launch();
  for (int i = tid; i <= p.E; i += kThreads) s_rdy[i] = 0;
  if (tid == 0) s_misc[0] = 0;  // routed experts: 0 until the routing is loaded
  __syncthreads();
  const Tables tb{s_off, s_act, s_sorted};

  const bool has_shared = p.Is > 0;
  const int nA_sh = has_shared ? p.Is / kSliceA : 0;
  const int nA_r = p.I / kSliceA;
  const int nB = p.H / kRowsB;
  const int fault = *(volatile int*)(p.hdr + kHdrFault);

  if (warp == kPW) {
    // ================================================================ producer
    // Lane 0 claims items, owns the ring and arms each stage's barrier; lanes
    // 0..3 issue the stage's tensor copies, lane tl the bulk copy of gathered
    // activation row tl.
    uint32_t gs = 0;         // stages issued
    int si = 0;              // ring slot of stage gs
    uint32_t ph = 0;         // parity of slot si's current use
    bool alive = true;
    int item = 0;
    bool all_ready = false;          // every w13 item (and every h group) is done
    // until the routing is loaded only the shared expert's w13 items are known
    bool routed = false;
    int totA = nA_sh, total = nA_sh;
    if (lane == 0) {
      // x codes and the reset counters of the router's first phase
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
    while (alive) {
      if (item >= nA_sh && !routed) {
        // the routing: the router grid has completed and its writes are visible
        // The tables (offsets, active experts: at most min(E, Mk), route order)
        // and the count come in one batch of independent loads: this hand-over
        // is on the layer's critical path.
        grid_dep_wait();
        const int nOff = p.E + 1, nAct = min(p.E, p.Mk), nAll = nOff + nAct + p.Mk;
        int n_act = 0;
        if (lane == 0) n_act = __ldcg(p.hdr + kHdrActive);
        for (int b0 = 0; b0 < nAll; b0 += 32 * kTabPer) {
          int v[kTabPer];
#pragma unroll
          for (int j = 0; j < kTabPer; ++j) {
            const int i = b0 + 32 * j + lane;
            v[j] = i < nOff ? __ldcg(p.off + i)
                 : i < nOff + nAct ? __ldcg(p.act + (i - nOff))
                 : i < nAll ? __ldcg(p.sorted + (i - nOff - nAct)) : 0;
          }
#pragma unroll
          for (int j = 0; j < kTabPer; ++j) {
            const int i = b0 + 32 * j + lane;
            if (i < nOff) s_off[i] = v[j];
            else if (i < nOff + nAct) s_act[i - nOff] = v[j];
            else if (i < nAll) s_sorted[i - nOff - nAct] = v[j];
          }
        }
        n_act = __shfl_sync(0xffffffffu, n_act, 0);
        if (lane == 0) s_misc[0] = n_act;  // for the epilogue warp's decoding
        __syncwarp();
        totA = nA_sh + n_act * nA_r;
        total = totA + ((has_shared ? 1 : 0) + n_act) * nB * (4 / p.bq);
        routed = true;
      }
      if (item >= total) break;
      int nxt = 0;
      if (lane == 0) nxt = atomicAdd(p.hdr + kHdrQueue, 1);
      const Item it = decode_item(item, nA_sh, nA_r, totA, nB, has_shared, p.bq);
      const Slot s = make_slot(p, tb, it.slot, has_shared);
      const int nkbK = it.a ? nkbH : s.Ie / kBlock;
      const int nkg = (nkbK + kKBS - 1) / kKBS;     // k-block groups
      const int nq = it.a ? 1 : p.bq;               // row quarters (B)
      const int nstage = nkg * nq;
      bool skip = false;
      // (lane 0 loads the counts below with ld.acquire, so that its later
      // reads, and the lanes' copies after the warp barrier, see what the
      // counted epilogues published; a generic-to-async proxy fence then
      // orders the TMA reads of h after them)
      if (!it.a && !all_ready) {
        // all w13 work done (lane 0's acquire of the count): covers every expert
        // from now on.  (Loading this count and the next expert's a stage ahead,
        // mid-item, measured 1.3% slower at 8 tokens: the acquires stall the
        // copies of the item in flight.)
        int done = 0;
        if (lane == 0) done = ld_acquire(p.hdr + kHdrDoneA);
        if (__shfl_sync(0xffffffffu, lane == 0 && done >= totA ? 1 : 0, 0)) {
          all_ready = true;
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
      }
      if (!it.a && !all_ready && !s_rdy[it.slot]) {
        // w2 items need the expert's quantised h: all of its groups
        int sk = 0;
        if (lane == 0) {
          const unsigned long long t0 = globaltimer_ns();
          for (long n = 0;; ++n) {
            if (ld_acquire(p.ready + it.slot) >= nkbK) break;
            if (*(volatile int*)status != 0 || n > (1l << 24)) { sk = 1; break; }
            if (globaltimer_ns() - t0 > kWaitNs) {
              atomicExch(status, MOE_ERR_DEVICE_TIMEOUT);
              sk = 1;
              break;
            }
            __nanosleep(64);
          }
          if (!sk) s_rdy[it.slot] = 1;
        }
        __syncwarp();  // the lanes' copies and scale reads come after lane 0's acquire
        asm volatile("fence.proxy.async.global;" ::: "memory");
        skip = __shfl_sync(0xffffffffu, sk, 0) != 0;
      }
      const int rg = kSliceA * it.idx;
      // weight-scale rows of the item's two 16-row tiles (w13: gate, up; w2: one block)
      const float* wsr0;
      const float* wsr1;
      if (it.a) {
        const float* base = s.e < 0 ? p.sw13_s : p.w13_s + (size_t)s.e * (2 * p.I / kBlock) * nkbH;
        wsr0 = base + (size_t)(rg / kBlock) * nkbH;
        wsr1 = base + (size_t)((s.Ie + rg) / kBlock) * nkbH;
      } else {
        wsr0 = wsr1 = (s.e < 0 ? p.sw2_s : p.w2_s + (size_t)s.e * nkbH * (p.I / kBlock)) + (size_t)it.idx * nkbK;
      }
      const int passes = skip ? 1 : (s.nt + kTok - 1) / kTok;
      for (int pass = 0; pass < passes && alive; ++pass) {
        const int ntok = min(kTok, s.nt - pass * kTok);
        // scale-row offset of this lane's token of the pass (x scales: w13, h scales: w2)
        int tok_off = 0;
        if (lane < ntok)
          tok_off = it.a ? token_of(p, tb, s, pass * kTok + lane) * nkbH : (s.hbase + pass * kTok + lane) * p.hsS;
        // activation rows: the shared expert's w13 items take the pass's x rows
        // as one TMA box per half; every other item one bulk copy per token
        // (lane tl: gathered x rows, or the expert's h rows), which at a few
        // tokens per expert moves only the rows that exist
        const bool xt = it.a && s.e < 0;
        const uint8_t* xsrc = nullptr;
        if (!xt && lane < ntok)
          xsrc = it.a ? p.xq + (size_t)token_of(p, tb, s, pass * kTok + lane) * p.H
                      : p.hq + (size_t)(s.hbase + pass * kTok + lane) * p.Imax;
        int qr = it.a ? 0 : it.q0, kb0 = 0;    // row quarter and first k-block of stage st
        for (int st = 0; st < (skip ? 1 : nstage); ++st) {
          int ok = 1;
          if (lane == 0) ok = mbar_wait(empty + si, ph ^ 1u, status);
          __syncwarp();  // the slot is rewritten only after the consumers released it
          if (!__shfl_sync(0xffffffffu, ok, 0)) { alive = false; break; }
          const int nkv = min(kKBS, nkbK - kb0);
          uint8_t* wdst = ring + (size_t)si * C::kSlot;
          uint8_t* xdst = wdst + kWBytes;
          int* md = meta + kMetaInts * si;
          if (st == 0 && !skip) {
            // the pass's scale rows, before the slot is armed
            if (lane < ntok) md[16 + lane] = tok_off;
            if (lane == 0) {
              *reinterpret_cast<const float**>(md + 8) = wsr0;
              *reinterpret_cast<const float**>(md + 10) = wsr1;
            }
            __syncwarp();
          }
          if (lane == 0) {
            const int fl = skip ? kSkip
                                : ((st == 0 ? kFirst : 0) | (kb0 + kKBS >= nkbK ? kLast : 0) |
                                   (st == nstage - 1 ? kPassEnd : 0) | (xt ? kXT : 0) | (it.a ? kA : 0));
            *reinterpret_cast<int4*>(md) = make_int4(item, pass | (qr << 16), kb0, fl);
            *reinterpret_cast<int2*>(md + 4) = make_int2(ntok, nkv);
            if (skip) mbar_arrive(full + si);
            else mbar_expect_tx(full + si, kWBytes + (xt ? 2 * C::kXHalf : ntok * nkv * kBlock));
          }
          __syncwarp();
          if (!skip) {
            if (!xt && lane < ntok)
              bulk_load(xdst + lane * kXStride, xsrc + (size_t)kb0 * kBlock, nkv * kBlock, full + si);
            // the stage's tensor copies, one per lane in one instruction: lanes 0/1
            // the two weight boxes [kb0, kb0 + 4) and [kb0 + 4, kb0 + 8), lanes 2/3
            // the matching activation boxes
            if (lane < 4) {
              const int h = lane & 1, kh = kb0 + h * kKH;
              if (lane < 2) {
                uint8_t* wd = wdst + h * kWHalf;
                if (it.a) {
                  if (s.e < 0) tma_load_5d(wd, &maps.sw13, 0, kh, rg, 0, 0, full + si);
                  else tma_load_5d(wd, &maps.w13, 0, kh, rg, 0, s.e, full + si);
                } else {
                  const int r0 = kRowsB * it.idx + kRowsQ * qr;
                  if (s.e < 0) tma_load_4d(wd, &maps.sw2, 0, kh, r0, 0, full + si);
                  else tma_load_4d(wd, &maps.w2, 0, kh, r0, s.e, full + si);
                }
              } else if (xt) {
                uint8_t* xd = xdst + h * C::kXHalf;
                if (it.a) tma_load_3d(xd, &maps.xq, 0, kh, pass * kTok, full + si);
                else tma_load_3d(xd, &maps.hq, 0, kh, s.hbase + pass * kTok, full + si);
              }
            }
          }
          ++gs;
          if (++si == nst) { si = 0; ph ^= 1u; }
          kb0 += kKBS;
          if (kb0 >= nkbK) { kb0 = 0; ++qr; }
        }
        __syncwarp();
      }
      item = __shfl_sync(0xffffffffu, nxt, 0);
    }
    // end marker, then make sure every copy this CTA issued has landed
    if (alive) {
      const int si = gs % nst;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(empty + si, ((gs / nst) & 1u) ^ 1u, status);
      if (__shfl_sync(0xffffffffu, ok, 0)) {
        if (lane == 0) {
          meta[kMetaInts * si + 3] = kEnd;
          mbar_arrive(full + si);
        }
        ++gs;
      }
    }
    // (every stage up to gs was armed and its copies issued in the same step;
    // the last nst of them are the only ones whose slots were not reused)
    if (lane == 0)
      for (uint32_t j = (gs > (uint32_t)nst ? gs - nst : 0); j < gs; ++j)
        mbar_wait_landed(full + (j % nst), (j / nst) & 1u, status);
    __syncwarp();
  } else if (warp == kEW) {
    // ================================================================ epilogue
    // Adds the k-block partial sums of each finished 32-row group, applies
    // SwiGLU (w13) or stores the rows (w2), and runs the group counters and the
    // re-quantisation of h, so the consumer warps never wait on global atomics.
    uint32_t uses = 0;
    int cur = -1;
    Item it{};
    Slot s{};
    while (true) {
      const int b = uses % C::kRedBufs, ph = (uses / C::kRedBufs) & 1;
      if (!mbar_wait(red_full + b, ph, status)) break;
      const int4 em = *reinterpret_cast<const int4*>(epi + 4 * b);
      if (em.w) break;  // end
      const float* rb = red + b * kRedF;
      const int item = em.x, pass = em.y & 0xffff, qr = em.y >> 16, flags = em.z;
      if (item != cur) {
        cur = item;
        // routed items come after the producer loaded the routing (and s_misc[0])
        const int totA = nA_sh + *(volatile int*)s_misc * nA_r;
        it = decode_item(item, nA_sh, nA_r, totA, nB, has_shared, p.bq);
        s = make_slot(p, tb, it.slot, has_shared);
      }
      const int ntok = min(kTok, s.nt - pass * kTok);
      if (it.a) {
        const int rg = kSliceA * it.idx;
        for (int idx = lane; idx < kSliceA * ntok; idx += 32) {
          const int i = idx % kSliceA, tl = idx / kSliceA;
          float gsum = 0.f, usum = 0.f;
#pragma unroll
          for (int w = 0; w < kKW; ++w) {
            gsum += rb[(0 * kKW + w) * 16 * kTok + i * kTok + tl];
            usum += rb[(1 * kKW + w) * 16 * kTok + i * kTok + tl];
          }
          const float z = fminf(gsum, p.limit);
          const float hv = z / (1.f + expf(-z)) * fminf(fmaxf(usum, -p.limit), p.limit);
          p.h[(size_t)(s.hbase + pass * kTok + tl) * p.Imax + rg + i] = hv;
        }
      } else {
        const int row0 = kRowsB * it.idx + kRowsQ * qr;
        for (int idx = lane; idx < kRowsQ * ntok; idx += 32) {
          const int rr = idx % kRowsQ, tl = idx / kRowsQ, n = pass * kTok + tl;
          float v = 0.f;
#pragma unroll
          for (int w = 0; w < kKW; ++w) v += rb[((rr >> 4) * kKW + w) * 16 * kTok + (rr & 15) * kTok + tl];
          float* dst = s.e < 0 ? p.shared_out + (size_t)n * p.H : p.rows + (size_t)tb.sorted[s.o + n] * p.H;
          dst[row0 + rr] = v;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(red_empty + b);
      ++uses;
      if (it.a && (flags & kPassEnd) && pass * kTok + kTok >= s.nt) {
        // the 8th finished slice of a 128-column group quantises the group
        int last = 0;
        if (lane == 0) {
          __threadfence();
          last = atomicAdd(p.gcount + it.slot * p.gI + it.idx / (kBlock / kSliceA), 1) == kBlock / kSliceA - 1;
        }
        if (__shfl_sync(0xffffffffu, last, 0)) {
          __threadfence();
          const int grp = it.idx / (kBlock / kSliceA);
          constexpr int kQB = 8;  // rows whose loads are in flight together
          for (int n0 = 0; n0 < s.nt; n0 += kQB) {
            float4 v[kQB];
#pragma unroll
            for (int j = 0; j < kQB; ++j)
              if (n0 + j < s.nt)
                v[j] = __ldcg(reinterpret_cast<const float4*>(p.h + (size_t)(s.hbase + n0 + j) * p.Imax +
                                                              grp * kBlock + 4 * lane));
#pragma unroll
            for (int j = 0; j < kQB; ++j) {
              if (n0 + j < s.nt) {
                const size_t row = (size_t)(s.hbase + n0 + j);
                const float amax =
                    warp_max(fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w))));
                const float scl = group_scale(amax, p.e8m0);
                *reinterpret_cast<uint32_t*>(p.hq + row * p.Imax + grp * kBlock + 4 * lane) =
                    f32x4_to_e4m3x4(__fdiv_rn(v[j].x, scl), __fdiv_rn(v[j].y, scl), __fdiv_rn(v[j].z, scl),
                                    __fdiv_rn(v[j].w, scl));
                if (lane == 0) p.hs[row * p.hsS + grp] = scl;
              }
            }
          }
          // the codes are read with TMA (async proxy) by other CTAs
          asm volatile("fence.proxy.async.global;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            __threadfence();
            if (!(fault && it.slot == 0)) atomicAdd(p.ready + it.slot, 1);
          }
        }
        if (lane == 0) atomicAdd(p.hdr + kHdrDoneA, 1);  // released by the fences above
      }
    }
  } else if (C::consumer(warp) >= 0) {
    // ================================================================ consumers
    const int cwi = C::consumer(warp);
    const int tile = cwi / kKW, kw = cwi % kKW;  // this warp's 16-row tile; k-blocks kw + j kKW, j < kKP
    // this thread's fragment offsets within a slot (A box [gu 2][row 16][kb 4][128 B]
    // for w13 tiles, B box [row 32][kb 4][128 B] for w2: either way row r of tile t
    // is 128-byte row (16 t + r) * 4 + k-block of its box; activation boxes
    // [token][kb 4][128 B]; bulk activation rows at a kXStride pitch)
    uint32_t a_off[kKP][2][2], xt_off[kKP][TT][2], xb_off[kKP][TT][2];
#pragma unroll
    for (int h = 0; h < kKP; ++h) {
      const int kl = h * kKW + kw, bx = kl / kKH, kk = kl % kKH;
#pragma unroll
      for (int sp = 0; sp < 2; ++sp) {
        a_off[h][sp][0] = bx * kWHalf + swz(0, (tile * 16 + g) * kKH + kk, q + 4 * sp);
        a_off[h][sp][1] = bx * kWHalf + swz(0, (tile * 16 + g + 8) * kKH + kk, q + 4 * sp);
      }
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const int tok = t * 8 + g;
        xt_off[h][t][0] = kWBytes + bx * C::kXHalf + swz(0, tok * kKH + kk, q);
        xt_off[h][t][1] = kWBytes + bx * C::kXHalf + swz(0, tok * kKH + kk, q + 4);
        xb_off[h][t][0] = kWBytes + tok * kXStride + kl * kBlock + q * 16;
        xb_off[h][t][1] = xb_off[h][t][0] + 64;
      }
    }
    const uint32_t ring_s = su32(ring);
    float acc[TT][4];
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
    uint32_t red_uses = 0;
    int si = 0;       // ring slot of the next stage
    uint32_t ph = 0;  // its parity
    const float* wsr = nullptr;   // this warp's weight-scale row (16-row tile's 128-row block)
    const float* xsr[TT][2];      // scale rows of this thread's token columns (or null)
    bool ok = true;
    while (true) {
      if (!mbar_wait(full + si, ph, status)) { ok = false; break; }
      const int* md = meta + kMetaInts * si;
      const int4 mt = *reinterpret_cast<const int4*>(md);
      const int item = mt.x, kb0 = mt.z, flags = mt.w;
      if (flags & kEnd) break;
      if (flags & kSkip) {
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + si);
        if (++si == nst) { si = 0; ph ^= 1u; }
        continue;
      }
      const int2 nn = *reinterpret_cast<const int2*>(md + 4);
      const int ntok = nn.x, nkv = nn.y;
      if (flags & kFirst) {
        // a new pass: its scale rows, as the producer resolved them
        wsr = *reinterpret_cast<const float* const*>(md + 8 + 2 * tile);
        const float* xbase = (flags & kA) ? p.xs : p.hs;
#pragma unroll
        for (int t = 0; t < TT; ++t)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int tl = t * 8 + 2 * q + j;
            xsr[t][j] = tl < ntok ? xbase + md[16 + tl] : nullptr;
          }
      }
      // block scales of this warp's k-blocks: issued first, used after the MMAs
      float wsc[kKP], xsc[kKP][TT][2];
#pragma unroll
      for (int h = 0; h < kKP; ++h) {
        const int kl = h * kKW + kw, kb = kb0 + kl;
        wsc[h] = kl < nkv ? ld_ca(wsr + kb) : 0.f;
#pragma unroll
        for (int t = 0; t < TT; ++t)
#pragma unroll
          for (int j = 0; j < 2; ++j) xsc[h][t][j] = (kl < nkv && xsr[t][j]) ? ld_ca(xsr[t][j] + kb) : 0.f;
      }

      // ---- this warp's tile of its k-blocks of the stage
      const uint32_t sb = ring_s + (uint32_t)si * C::kSlot;
      const bool xt = (flags & kXT) != 0;
#pragma unroll
      for (int h = 0; h < kKP; ++h) {
        if (h * kKW + kw < nkv) {
          uint4 a0[2], a1[2];
#pragma unroll
          for (int sp = 0; sp < 2; ++sp) {
            a0[sp] = lds128(sb + a_off[h][sp][0]);
            a1[sp] = lds128(sb + a_off[h][sp][1]);
          }
          const float ws = wsc[h];
#pragma unroll
          for (int t = 0; t < TT; ++t) {
            if (t * 8 < ntok) {  // token tiles past the pass do no work
              uint4 x0 = make_uint4(0, 0, 0, 0), x1 = x0;
              if (t * 8 + g < ntok) {
                x0 = lds128(sb + (xt ? xt_off[h][t][0] : xb_off[h][t][0]));
                x1 = lds128(sb + (xt ? xt_off[h][t][1] : xb_off[h][t][1]));
              }
              float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
              mma_span_e4m3(c0, a0[0], a1[0], x0);
              mma_span_e4m3(c1, a0[1], a1[1], x1);
              // token columns past the pass have scale 0
              const float f0 = ws * xsc[h][t][0], f1 = ws * xsc[h][t][1];
              acc[t][0] += (c0[0] + c1[0]) * f0;
              acc[t][1] += (c0[1] + c1[1]) * f1;
              acc[t][2] += (c0[2] + c1[2]) * f0;
              acc[t][3] += (c0[3] + c1[3]) * f1;
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + si);
      if (++si == nst) { si = 0; ph ^= 1u; }

      if (flags & kLast) {
        // ---- hand this 32-row group's partial sums to the epilogue warp
        const int b = red_uses % C::kRedBufs;
        if (!mbar_wait(red_empty + b, ((red_uses / C::kRedBufs) & 1u) ^ 1u, status)) { ok = false; break; }
        float* r = red + b * kRedF + (tile * kKW + kw) * 16 * kTok;
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          if (t * 8 < ntok) {
            const int tl = t * 8 + 2 * q;
            r[g * kTok + tl] = acc[t][0];
            r[g * kTok + tl + 1] = acc[t][1];
            r[(g + 8) * kTok + tl] = acc[t][2];
            r[(g + 8) * kTok + tl + 1] = acc[t][3];
          }
          acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
        }
        if (cwi == 0 && lane == 0) *reinterpret_cast<int4*>(epi + 4 * b) = make_int4(item, mt.y, flags, 0);
        __syncwarp();
        if (lane == 0) mbar_arrive(red_full + b);
        ++red_uses;
      }
    }
    // tell the epilogue warp to finish (in the next hand-off buffer, once free)
    const int b = red_uses % C::kRedBufs;
    if (ok && mbar_wait(red_empty + b, ((red_uses / C::kRedBufs) & 1u) ^ 1u, status)) {
      if (cwi == 0 && lane == 0) *reinterpret_cast<int4*>(epi + 4 * b) = make_int4(0, 0, 0, 1);
      __syncwarp();
      if (lane == 0) mbar_arrive(red_full + b);
    }
  }
  __syncthreads();
  if (tid == 0) {
    // the last CTA to finish clears the router's x-ready count for the next call
    // (every CTA has passed its wait on it; the next router starts after this grid)
    __threadfence();
    if (atomicAdd(p.hdr + kHdrExit, 1) == (int)gridDim.x - 1) {
      p.hdr[kHdrXReady] = 0;
      p.hdr[kHdrExit] = 0;
    }
  }
}

// ------------------------------------------------------------- host side
}  // namespace

EncodeTiledFn encode_fn() {
  // looked up once (a thread-safe static initialisation)
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

bool tmap_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols, uint32_t box_rows) {
  if (!encode_fn()) return false;
  const cuuint64_t dim[2] = {cols, rows};
  const cuuint64_t stride[1] = {cols};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dim, stride, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// w13 of n experts as [n][2][I][H/128][128] bytes; box = 16 rows of gate and up
// x 4 k-blocks x 128 bytes.
bool map_w13(CUtensorMap* m, const uint8_t* base, int H, int I, int n) {
  const cuuint64_t dim[5] = {128, (cuuint64_t)H / 128, (cuuint64_t)I, 2, (cuuint64_t)n};
  const cuuint64_t stride[4] = {128, (cuuint64_t)H, (cuuint64_t)I * H, (cuuint64_t)2 * I * H};
  const cuuint32_t box[5] = {128, kKH, kSliceA, 2, 1};
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<uint8_t*>(base), dim, stride, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// w2 of n experts as [n][H][I/128][128]; box = 32 rows x 4 k-blocks x 128 bytes.
bool map_w2(CUtensorMap* m, const uint8_t* base, int H, int I, int n) {
  const cuuint64_t dim[4] = {128, (cuuint64_t)I / 128, (cuuint64_t)H, (cuuint64_t)n};
  const cuuint64_t stride[3] = {128, (cuuint64_t)I, (cuuint64_t)H * I};
  const cuuint32_t box[4] = {128, kKH, kRowsQ, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t*>(base), dim, stride, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int TT>
size_t other_smem(const ExpertArgs& a, int nst) {
  return (size_t)nst * (Cfg<TT>::kMetaInts * sizeof(int) + 2 * sizeof(uint64_t)) + 2 * sizeof(uint64_t) + 4 * sizeof(int) +
         sizeof(float) * ((size_t)Cfg<TT>::kRedBufs * 2 * Cfg<TT>::kKW * 16 * Cfg<TT>::kTok) + 4 * sizeof(int) +
         2 * sizeof(uint64_t) +
         sizeof(int) * (3 * a.E + 2 + a.Mk + 4) + 1024;
}

// activation codes [rows][K/128][128] bytes; box = 4 k-blocks x `box_rows` rows
bool map_rows(CUtensorMap* m, const uint8_t* base, int K, int rows, int box_rows) {
  const cuuint64_t dim[3] = {128, (cuuint64_t)K / 128, (cuuint64_t)rows};
  const cuuint64_t stride[2] = {128, (cuuint64_t)K};
  const cuuint32_t box[3] = {128, kKH, (cuuint32_t)box_rows};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(base), dim, stride, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int TT>
cudaError_t prepare_tt(const ExpertArgs& a, ExpertsLaunch& L) {
  TmaMaps* maps = reinterpret_cast<TmaMaps*>(L.maps);
  if (!map_rows(&maps->xq, a.xq, a.H, a.M, Cfg<TT>::kTok) ||
      !map_rows(&maps->hq, a.hq, a.Imax, a.Mk + a.M, Cfg<TT>::kTok))
    return cudaErrorInvalidValue;
  int nst = Cfg<TT>::kNSTMax;
  while (nst > 2 && (size_t)nst * Cfg<TT>::kSlot + other_smem<TT>(a, nst) > (size_t)kSmemMax) --nst;
  const size_t smem = (size_t)nst * Cfg<TT>::kSlot + other_smem<TT>(a, nst);
  if (smem > (size_t)kSmemMax) return cudaErrorInvalidConfiguration;
  L.tt = TT;
  L.nst = nst;
  L.smem = smem;
  return cudaFuncSetAttribute(experts_kernel<TT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

template <int TT>
cudaError_t launch_tt(const ExpertsLaunch& L, int num_sms, cudaStream_t s) {
  TmaMaps maps;
  memcpy(&maps, L.maps, sizeof(maps));
  PdlLaunch P(dim3(num_sms), dim3(Cfg<TT>::kThreads), L.smem, s);
  return cudaLaunchKernelEx(&P.cfg, experts_kernel<TT>, L.a, maps, L.nst);
}

}  // namespace

static_assert(sizeof(TmaMaps) <= sizeof(ExpertsLaunch::maps), "tensor maps fit the prepared launch");

cudaError_t launch_experts_tc_prepared(const ExpertsLaunch& L, int num_sms, cudaStream_t s);

cudaError_t prepare_experts(const ExpertArgs& a, ExpertsLaunch& L) {
  if (!encode_fn()) return cudaErrorNotSupported;
  memset(&L, 0, sizeof(L));
  L.a = a;
  L.tc = false;
  TmaMaps* maps = reinterpret_cast<TmaMaps*>(L.maps);
  // (a dense layer has no routed experts: their maps stay zero, never used)
  if (a.E > 0 && (!map_w13(&maps->w13, a.w13, a.H, a.I, a.E) || !map_w2(&maps->w2, a.w2, a.H, a.I, a.E)))
    return cudaErrorInvalidValue;
  if (a.Is > 0 && (!map_w13(&maps->sw13, a.sw13, a.H, a.Is, 1) || !map_w2(&maps->sw2, a.sw2, a.H, a.Is, 1)))
    return cudaErrorInvalidValue;
  // Passes of 8 tokens: an expert with more tokens (the shared expert above
  // M = 8) streams its rows once per pass, the repeats from L2.  Wider passes
  // cost consumer registers and ring stages, and measured slower on the
  // DeepSeek-V3-shaped layer up to M = 128 tokens; 16-token passes win above.
  if (a.E == 0) {
    // a dense layer: every token goes through the one MLP, so the widest pass
    // streams its weights the fewest times
    if (a.M <= 8) return prepare_tt<1>(a, L);
    if (a.M <= 16) return prepare_tt<2>(a, L);
    return prepare_tt<4>(a, L);
  }
  if (a.M <= 128) return prepare_tt<1>(a, L);
  return prepare_tt<2>(a, L);
}

cudaError_t launch_experts(const ExpertsLaunch& L, int num_sms, cudaStream_t s) {
  if (L.tc) return launch_experts_tc_prepared(L, num_sms, s);
  switch (L.tt) {
    case 1: return launch_tt<1>(L, num_sms, s);
    case 2: return launch_tt<2>(L, num_sms, s);
    default: return launch_tt<4>(L, num_sms, s);
  }
}

}  // namespace moe
