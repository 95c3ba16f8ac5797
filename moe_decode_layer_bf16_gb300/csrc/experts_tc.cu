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
constexpr int kPW = 0, kMW = 1, kEW0 = 4, kNEpi = 8;
constexpr int kSegKB = 16;               // k-blocks of a w2 item's K segment, when I is split

static_assert(kNST * 2 * kPass == kTCols, "one accumulator pair per ring stage");

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
// 32 consecutive fp32 columns of this thread's lane
MOE_DEV void tc_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// Bounded wait that ignores the status word (the waits of the MMA and
// epilogue warps end together, by the phase or by the bound).
MOE_DEV bool mbar_wait_t(uint64_t* b, uint32_t parity, int* status) { return mbar_wait_landed(b, parity, status); }

// ------------------------------------------------------------- work items
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

MOE_DEV TcItem tc_decode(int item, int nA_sh, int nA_r, int totA, int nB, int sh_segs, bool has_shared) {
  TcItem it;
  if (item < totA) {
    it.a = true;
    it.seg = 0;
    if (item < nA_sh) {
      it.slot = 0;
      it.idx = item;
    } else {
      const int j = item - nA_sh;
      it.slot = j / nA_r + (has_shared ? 1 : 0);
      it.idx = j % nA_r;
    }
  } else {
    it.a = false;
    int j = item - totA;
    const int nBs = has_shared ? nB * sh_segs : 0;
    if (j < nBs) {
      it.slot = 0;
      it.idx = j / sh_segs;
      it.seg = j % sh_segs;
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

// K range of an item, in k-blocks: all of H (A) or segment seg of Ie (B)
MOE_DEV void tc_krange(const ExpertArgs& p, const TcItem& it, const TcSlot& s, int sh_segs, int& k0, int& k1) {
  if (it.a) {
    k0 = 0;
    k1 = p.H / kBlock;
    return;
  }
  const int nkb = s.Ie / kBlock;
  const int segs = s.e < 0 ? sh_segs : 1;
  const int len = (nkb + segs - 1) / segs;
  k0 = it.seg * len;
  k1 = min(nkb, k0 + len);
}

struct TcMaps {
  CUtensorMap w13, w2, sw13, sw2;  // weights, box 128 B x 128 rows
  CUtensorMap xq;                  // x codes [M][H], box 128 B x 16 rows
  CUtensorMap xg;                  // routed x codes gathered in route order [Mk][H]
  CUtensorMap hq;                  // h codes [Mk + M][Imax]
};

struct TcArgs {
  const uint8_t* xg;
  int sh_segs;  // K segments of the shared slot's w2 items (partial rows the boundary adds)
};

__global__ void __launch_bounds__(kThreads, 1)
    experts_tc_kernel(ExpertArgs p, TcArgs q, const __grid_constant__ TcMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (su32(smem_raw) & 1023)) & 1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nkbH = p.H / kBlock;

  // ---- shared memory: ring | stage descriptors | accumulator descriptors | barriers | epilogue buffers | tables
  uint8_t* ring = smem;
  int* meta = reinterpret_cast<int*>(smem + (size_t)kNST * kSlotB);   // [kNST][kMetaInts]
  int* tmeta = meta + kNST * kMetaInts;                                  // [kNST][kMetaInts]
  uint64_t* full = reinterpret_cast<uint64_t*>(tmeta + kNST * kMetaInts);
  uint64_t* empty = full + kNST;
  uint64_t* tfull = empty + kNST;
  uint64_t* tempty = tfull + kNST;
  uint64_t* amax_bar = tempty + kNST;   // [2 pass parities][2 column halves]
  uint64_t* mma_done = amax_bar + 4;
  float* cbuf = reinterpret_cast<float*>(mma_done + 2);                 // [8 warps][2][32]
  float* amax_buf = cbuf + kNEpi * 64;                                   // [2][2][4][32]
  int* s_misc = reinterpret_cast<int*>(amax_buf + 2 * 2 * 4 * 32);       // [0] tensor-memory base, [1] routed experts
  int* s_off = s_misc + 4;                                               // [E+1]
  int* s_act = s_off + (p.E + 1);                                        // [E]
  int* status = p.hdr + kHdrStatus;

  if (tid == 0) {
    for (int i = 0; i < kNST; ++i) {
      mbar_init(full + i, 1);    // the producer's expect-tx arrival
      mbar_init(empty + i, 2);   // the MMAs' commit + the MMA thread
      mbar_init(tfull + i, 2);   // the MMAs' commit + the MMA thread
      mbar_init(tempty + i, kNEpi);
    }
    for (int i = 0; i < 4; ++i) mbar_init(amax_bar + i, 4);
    mbar_init(mma_done, 1);
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
  const int nA_sh = has_shared ? p.Is / kRows : 0;
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
      int nxt = 0;
      if (lane == 0) nxt = atomicAdd(p.hdr + kHdrQueue, 1);
      const TcItem it = tc_decode(item, nA_sh, nA_r, totA, nB, q.sh_segs, has_shared);
      const TcSlot s = tc_slot(p, s_off, s_act, it.slot, has_shared);
      int k0, k1;
      tc_krange(p, it, s, q.sh_segs, k0, k1);
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
      for (int pass = 0; pass < passes && alive; ++pass) {
        const int ntok = min(kPass, s.nt - pass * kPass);
        const int npad = (ntok + 15) & ~15;
        // activation rows of the pass: x rows (shared expert, dense), gathered
        // x rows in route order (routed), h rows (w2)
        const CUtensorMap* xmap = it.a ? (s.e < 0 ? &maps.xq : &maps.xg) : &maps.hq;
        const int xrow = (it.a ? (s.e < 0 ? 0 : s.o) : s.hbase) + pass * kPass;
        for (int kb = k0; kb < k1; kb += kstep) {
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
      item = __shfl_sync(0xffffffffu, nxt, 0);
    }
    // end marker, then make sure every copy this CTA issued has landed
    {
      int ok = 1;
      if (lane == 0) ok = mbar_wait_landed(empty + si, ph ^ 1u, status);
      if (__shfl_sync(0xffffffffu, ok, 0)) {
        if (lane == 0) {
          meta[kMetaInts * si + 3] = kFEnd;
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
  } else if (warp >= kEW0) {
    // ================================================================ epilogue
    const int ew = warp - kEW0;
    const int qd = warp & 3;           // tensor-memory lane quadrant: rows 32 qd .. 32 qd + 31
    const int hf = ew >> 2;            // token column half: columns 32 hf .. 32 hf + 31 of a pass
    const int col0 = 32 * hf;
    const int r = 32 * qd + lane;      // this thread's row of the 128-row tile
    float* cb = cbuf + ew * 64;
    float acc0[32], acc1[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) acc0[j] = acc1[j] = 0.f;
    int cur_item = -1, cur_pass = -1;
    TcItem it{};
    TcSlot s{};
    const float* ws0 = nullptr;  // weight-scale rows: A gate / up, B the 128-row block
    const float* ws1 = nullptr;
    const float* xsr = nullptr;  // this lane's token's scale row (A: x, B: h), null past the pass
    int out_row = 0;             // B: this lane's token's output row
    uint32_t pe = 0;  // A-item pass ends so far: the amax buffer and barrier alternate with it
    int si = 0;
    uint32_t ph = 0;
    while (true) {
      if (!mbar_wait_t(tfull + si, ph, status)) break;
      const int* tm = tmeta + kMetaInts * si;
      const int4 m0 = *reinterpret_cast<const int4*>(tm);
      const int4 m1 = *reinterpret_cast<const int4*>(tm + 4);
      if (m0.w & kFEnd) break;
      const int item = m0.x, pass = m0.y, kb = m0.z, fl = m0.w, ntok = m1.x, nkv = m1.z;
      const bool a = (fl & kFA) != 0;
      if (item != cur_item) {
        cur_item = item;
        cur_pass = -1;
        // routed items come after the producer loaded the routing tables
        const int n_act = *(volatile int*)(s_misc + 1);
        const int totA = nA_sh + n_act * nA_r;
        it = tc_decode(item, nA_sh, nA_r, totA, nB, q.sh_segs, has_shared);
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
        const int tl = pass * kPass + col0 + lane;  // this lane's token of the slot
        xsr = nullptr;
        if (col0 + lane < ntok) {
          if (a) {
            const int tok = s.e < 0 ? tl : __ldcg(p.sorted + s.o + tl) / p.k;
            xsr = p.xs + (size_t)tok * nkbH;
          } else {
            xsr = p.hs + (size_t)(s.hbase + tl) * p.hsS;
            out_row = s.e < 0 ? tl : __ldcg(p.sorted + s.o + tl);
          }
        }
      }
      const bool mine = col0 < ntok;  // this warp's columns hold tokens of the pass
      if (mine) {
        // scale of each column: weight block scale x token group scale (x
        // scales through L1; h scales from L2, since a split w2 item may meet
        // a line whose other groups another CTA writes later)
        float c0, c1;
        if (a) {
          const float sx = xsr ? ld_ca(xsr + kb) : 0.f;
          c0 = ld_ca(ws0 + kb) * sx;
          c1 = ld_ca(ws1 + kb) * sx;
        } else {
          c0 = xsr ? ld_ca(ws0 + kb) * __ldcg(xsr + kb) : 0.f;
          c1 = (xsr && nkv > 1) ? ld_ca(ws0 + kb + 1) * __ldcg(xsr + kb + 1) : 0.f;
        }
        cb[lane] = c0;
        cb[32 + lane] = c1;
        __syncwarp();
      }
      tc_fence_after();
      if (mine) {
        const uint32_t ta = tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(si * 2 * kPass + col0);
        float d[32];
        tc_ld32(ta, d);
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          const float4 f0 = *reinterpret_cast<const float4*>(cb + j);
          acc0[j] += d[j] * f0.x; acc0[j + 1] += d[j + 1] * f0.y;
          acc0[j + 2] += d[j + 2] * f0.z; acc0[j + 3] += d[j + 3] * f0.w;
        }
        if (a) {
          tc_ld32(ta + kPass, d);  // the up rows
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 f1 = *reinterpret_cast<const float4*>(cb + 32 + j);
            acc1[j] += d[j] * f1.x; acc1[j + 1] += d[j + 1] * f1.y;
            acc1[j + 2] += d[j + 2] * f1.z; acc1[j + 3] += d[j + 3] * f1.w;
          }
        } else if (nkv > 1) {
          tc_ld32(ta + kPass, d);  // the stage's second k-block
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 f1 = *reinterpret_cast<const float4*>(cb + 32 + j);
            acc0[j] += d[j] * f1.x; acc0[j + 1] += d[j + 1] * f1.y;
            acc0[j + 2] += d[j + 2] * f1.z; acc0[j + 3] += d[j + 3] * f1.w;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty + si);
      if (++si == kNST) { si = 0; ph ^= 1u; }
      if (!(fl & kFLast)) continue;

      // ---- end of a pass
      const int nval = min(32, max(0, ntok - col0));  // this warp's token columns
      const int tl0 = pass * kPass + col0;
      if (!a) {
        // w2: this thread's row of every token's output (fp32), unweighted
        const int hrow = kRows * it.idx + r;
        float* base = s.e < 0 ? p.shared_out + (size_t)it.seg * p.M * p.H : p.rows;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int orow = __shfl_sync(0xffffffffu, out_row, j);
          if (j < nval) base[(size_t)orow * p.H + hrow] = acc0[j];
        }
      } else {
        // w13: h = silu(min(g, L)) * clamp(u, -L, L), then FP8 per token over the
        // 128 intermediates of this item (the four lane quadrants of the column half)
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float z = fminf(acc0[j], p.limit);
          acc0[j] = z / (1.f + expf(-z)) * fminf(fmaxf(acc1[j], -p.limit), p.limit);
          acc1[j] = j < nval ? fabsf(acc0[j]) : 0.f;
        }
        // per-column max over this warp's 32 rows: after the five exchange
        // steps lane l holds the max of column l
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
        const int grp = it.idx;  // the item's 128 intermediates are h group idx
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float sj = __shfl_sync(0xffffffffu, scl, j);
          if (j < nval) {
            const size_t row = (size_t)(s.hbase + tl0 + j);
            uint16_t code;
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(code) : "f"(0.f), "f"(__fdiv_rn(acc0[j], sj)));
            p.hq[row * p.Imax + grp * kBlock + r] = (uint8_t)(code & 0xff);
          }
        }
        if (qd == 0 && lane < nval) p.hs[(size_t)(s.hbase + tl0 + lane) * p.hsS + grp] = scl;
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

size_t tc_smem_bytes(int E) {
  return 1024 + (size_t)kNST * kSlotB + 2 * kNST * kMetaInts * sizeof(int) +
         (4 * kNST + 4 + 2) * sizeof(uint64_t) + (kNEpi * 64 + 2 * 2 * 4 * 32) * sizeof(float) +
         (4 + 2 * E + 1) * sizeof(int);
}

}  // namespace

int tc_shared_segments(int Is, int M) {
  // a dense layer's long w2 rows (I_s / 128 k-blocks) are split into segments
  // of 16 k-blocks while one pass holds all tokens, so that the w2 phase has
  // enough items for every SM; the boundary adds the partial rows
  if (Is <= 0 || M > kPass) return 1;
  return std::max(1, (Is / kBlock + kSegKB - 1) / kSegKB);
}

cudaError_t launch_experts_tc(const ExpertArgs& a, const uint8_t* xg, int sh_segs, int num_sms, cudaStream_t s) {
  if (!encode_fn()) return cudaErrorNotSupported;
  TcMaps maps;
  memset(&maps, 0, sizeof(maps));
  // weights: [rows][K] bytes, box one k-block x 128 rows; activations box one k-block x 16 rows
  if (a.E > 0 && (!tmap_2d(&maps.w13, a.w13, a.H, (uint64_t)a.E * 2 * a.I, 128, kRows) ||
                  !tmap_2d(&maps.w2, a.w2, a.I, (uint64_t)a.E * a.H, 128, kRows) ||
                  !tmap_2d(&maps.xg, xg, a.H, a.Mk, 128, 16)))
    return cudaErrorInvalidValue;
  if (a.Is > 0 && (!tmap_2d(&maps.sw13, a.sw13, a.H, 2 * (uint64_t)a.Is, 128, kRows) ||
                   !tmap_2d(&maps.sw2, a.sw2, a.Is, a.H, 128, kRows)))
    return cudaErrorInvalidValue;
  if (!tmap_2d(&maps.xq, a.xq, a.H, a.M, 128, 16) || !tmap_2d(&maps.hq, a.hq, a.Imax, (uint64_t)a.Mk + a.M, 128, 16))
    return cudaErrorInvalidValue;
  const size_t smem = tc_smem_bytes(a.E);
  if (smem > 227 * 1024) return cudaErrorInvalidConfiguration;
  cudaError_t err = cudaFuncSetAttribute(experts_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  TcArgs q;
  q.xg = xg;
  q.sh_segs = sh_segs;
  PdlLaunch L(dim3(num_sms), dim3(kThreads), smem, s);
  return cudaLaunchKernelEx(&L.cfg, experts_tc_kernel, a, q, maps);
}

cudaError_t launch_gather_rows(const uint8_t* xq, const int* sorted, int k, int Mk, int H, uint8_t* xg, int num_sms,
                               cudaStream_t s) {
  if (Mk <= 0) return cudaSuccess;
  PdlLaunch L(dim3(std::min(Mk, 2 * num_sms)), dim3(256), 0, s);
  return cudaLaunchKernelEx(&L.cfg, gather_rows_kernel, xq, sorted, k, Mk, H, xg);
}

}  // namespace moe
