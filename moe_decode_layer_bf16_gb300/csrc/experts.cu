// The routed + shared experts of one MoE decode step as one persistent kernel
// (the decode page, vllm.models.glm5next.nvidia.specialized_decode.runtime
// .decode, LayerStages._mega_moe: "routed experts as one kernel"; its grouped
// form "runs the shared expert as one more expert", which is what this kernel
// does at every token count).
//
// Per expert: [g; u] = xq . w13^T with 128x128 block scales, clamped SwiGLU
// h = silu(min(g, L)) * clamp(u, -L, L), h re-quantised to FP8 per route per
// 128-column group, y = hq . w2^T.  Routed outputs are written unweighted, in
// expanded route order (the page's UnfinalizedMoEOutput rows with the
// identity expanded->permuted map); the shared expert's output separately.
//
// Work: the decode step streams each active expert's FP8 weights exactly once
// and is HBM-bound at every token count this layer sees, so the kernel is a
// balanced weight stream:
//   A items (expert, 16 intermediates): 16 gate + 16 up rows of w13 over all
//     of H, split over the CTA's 4 warps by k-block, reduced in shared memory;
//   B items (expert, 64 rows of w2) over all of I, one 16-row tile per warp.
// A CTA pulls items from one queue (all A items, then all B items).  The A
// item that completes the 8th slice of a 128-column group quantises that
// group for every route; an expert's B items start once all of its groups are
// quantised (a bounded wait: after ~0.2 s it records MOE_ERR_DEVICE_TIMEOUT
// in the workspace status word and skips the item, so the kernel always ends).
// Only items already taken by running CTAs are ever waited on, so the queue
// cannot deadlock however many CTAs are resident.
//
// Each warp streams its operands through a private ring of cp.async stages
// (16-byte copies, L1 bypassed), and the products run on warp-level FP8 MMAs
// (m16n8k32, fp32 accumulate).  Per 128-column block the MMA sum is scaled by
// weight scale x activation scale and added to fp32 accumulators.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "../../include/moe_decode.h"

namespace moe {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kNST = 3;            // cp.async stages per warp
constexpr int kSliceA = 16;        // intermediates per A item
constexpr int kRowsB = 64;         // w2 rows per B item
constexpr unsigned long long kWaitNs = 200ull * 1000ull * 1000ull;

template <int TT>
struct Cfg {
  static constexpr int kTok = 8 * TT;                // tokens per pass
  static constexpr int kStageW = 8 * 512;            // 8 chunks of 16 B per lane
  static constexpr int kStage = kStageW + 2 * TT * 512;
  static constexpr int kRingWarp = kNST * kStage;
  static constexpr int kRing = kWarps * kRingWarp;
};

MOE_DEV void cp_async16(void* smem, const void* gmem, bool valid) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}
MOE_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
MOE_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

struct Slot {
  const uint8_t* w13; const float* s13;
  const uint8_t* w2; const float* s2;
  int Ie;      // intermediate size of this expert
  int nt;      // routes (tokens) of this expert
  int o;       // first position in the sorted route list (routed)
  int hbase;   // first h row
  bool shared;
};

struct Smem {
  int* off;     // [E+1]
  int* act;     // [E]
  int* sorted;  // [Mk]
  float* sc;    // activation scales of a pass [kTok][nkb]
  float* sw;    // weight scales [2][nkb]
  uint8_t* ring;
};

MOE_DEV int token_of(const ExpertArgs& p, const Smem& sm, const Slot& s, int i) {
  return s.shared ? i : sm.sorted[s.o + i] / p.k;
}

MOE_DEV Slot make_slot(const ExpertArgs& p, const Smem& sm, int slot, bool has_shared) {
  Slot s;
  if (has_shared && slot == 0) {
    s.w13 = p.sw13; s.s13 = p.sw13_s; s.w2 = p.sw2; s.s2 = p.sw2_s;
    s.Ie = p.Is; s.nt = p.M; s.o = 0; s.hbase = p.Mk; s.shared = true;
  } else {
    const int e = sm.act[slot - (has_shared ? 1 : 0)];
    const size_t nkbH = p.H / kBlock;
    s.w13 = p.w13 + (size_t)e * 2 * p.I * p.H;
    s.s13 = p.w13_s + (size_t)e * (2 * p.I / kBlock) * nkbH;
    s.w2 = p.w2 + (size_t)e * p.H * p.I;
    s.s2 = p.w2_s + (size_t)e * nkbH * (p.I / kBlock);
    s.Ie = p.I; s.o = sm.off[e]; s.nt = sm.off[e + 1] - s.o; s.hbase = s.o; s.shared = false;
  }
  return s;
}

// ------------------------------------------------------------------ A item
template <int TT>
__device__ void run_A(const ExpertArgs& p, const Smem& sm, const Slot& s, int slot, int sl, int fault) {
  using C = Cfg<TT>;
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, q = lane & 3;
  const int nkb = p.H / kBlock;
  const int kb_lo = warp * nkb / kWarps, kb_hi = (warp + 1) * nkb / kWarps, nk = kb_hi - kb_lo;
  const size_t H = p.H;
  const int rg = kSliceA * sl, ru = s.Ie + kSliceA * sl;
  const uint8_t* wg0 = s.w13 + (size_t)(rg + g) * H + 16 * q;
  const uint8_t* wg1 = wg0 + 8 * H;
  const uint8_t* wu0 = s.w13 + (size_t)(ru + g) * H + 16 * q;
  const uint8_t* wu1 = wu0 + 8 * H;
  uint8_t* ring = sm.ring + warp * C::kRingWarp;

  for (int p0 = 0; p0 < s.nt; p0 += C::kTok) {
    int tokB[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      const int n = p0 + t * 8 + g;
      tokB[t] = n < s.nt ? token_of(p, sm, s, n) : -1;
    }
    auto issue = [&](int kb, int st) {
      uint8_t* b = ring + st * C::kStage;
      const size_t ko = (size_t)kb * kBlock;
      cp_async16(b + (0 * 32 + lane) * 16, wg0 + ko, true);
      cp_async16(b + (1 * 32 + lane) * 16, wg0 + ko + 64, true);
      cp_async16(b + (2 * 32 + lane) * 16, wg1 + ko, true);
      cp_async16(b + (3 * 32 + lane) * 16, wg1 + ko + 64, true);
      cp_async16(b + (4 * 32 + lane) * 16, wu0 + ko, true);
      cp_async16(b + (5 * 32 + lane) * 16, wu0 + ko + 64, true);
      cp_async16(b + (6 * 32 + lane) * 16, wu1 + ko, true);
      cp_async16(b + (7 * 32 + lane) * 16, wu1 + ko + 64, true);
      uint8_t* xb = b + C::kStageW;
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const uint8_t* src = p.xq + (size_t)(tokB[t] < 0 ? 0 : tokB[t]) * H + ko + 16 * q;
        cp_async16(xb + ((2 * t) * 32 + lane) * 16, src, tokB[t] >= 0);
        cp_async16(xb + ((2 * t + 1) * 32 + lane) * 16, src + 64, tokB[t] >= 0);
      }
    };
#pragma unroll
    for (int i = 0; i < kNST - 1; ++i) {
      if (i < nk) issue(kb_lo + i, i);
      cp_async_commit();
    }
    // block scales of this pass: activation [kTok][nkb], weight gate/up [nkb]
    for (int idx = tid; idx < C::kTok * nkb; idx += kThreads) {
      const int n = p0 + idx / nkb, kb = idx % nkb;
      sm.sc[idx] = n < s.nt ? __ldg(p.xs + (size_t)token_of(p, sm, s, n) * nkb + kb) : 0.f;
    }
    for (int kb = tid; kb < nkb; kb += kThreads) {
      sm.sw[kb] = __ldg(s.s13 + (size_t)(rg / kBlock) * nkb + kb);
      sm.sw[nkb + kb] = __ldg(s.s13 + (size_t)(ru / kBlock) * nkb + kb);
    }
    __syncthreads();

    float ag[TT][4], au[TT][4];
#pragma unroll
    for (int t = 0; t < TT; ++t)
#pragma unroll
      for (int j = 0; j < 4; ++j) ag[t][j] = au[t][j] = 0.f;

#pragma unroll 1
    for (int i = 0; i < nk; ++i) {
      {
        const int j = i + kNST - 1;
        if (j < nk) issue(kb_lo + j, j % kNST);
        cp_async_commit();
      }
      cp_async_wait<kNST - 1>();
      const uint4* b = reinterpret_cast<const uint4*>(ring + (i % kNST) * C::kStage);
      const uint4 g00 = b[0 * 32 + lane], g01 = b[1 * 32 + lane];
      const uint4 g10 = b[2 * 32 + lane], g11 = b[3 * 32 + lane];
      const uint4 u00 = b[4 * 32 + lane], u01 = b[5 * 32 + lane];
      const uint4 u10 = b[6 * 32 + lane], u11 = b[7 * 32 + lane];
      const int kb = kb_lo + i;
      const float swg = sm.sw[kb], swu = sm.sw[nkb + kb];
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const uint4 x0 = b[(8 + 2 * t) * 32 + lane], x1 = b[(9 + 2 * t) * 32 + lane];
        float cg[4] = {0.f, 0.f, 0.f, 0.f}, cu[4] = {0.f, 0.f, 0.f, 0.f};
        mma_span_e4m3(cg, g00, g10, x0);
        mma_span_e4m3(cg, g01, g11, x1);
        mma_span_e4m3(cu, u00, u10, x0);
        mma_span_e4m3(cu, u01, u11, x1);
        const float sx0 = sm.sc[(t * 8 + 2 * q) * nkb + kb], sx1 = sm.sc[(t * 8 + 2 * q + 1) * nkb + kb];
        const float fg0 = swg * sx0, fg1 = swg * sx1, fu0 = swu * sx0, fu1 = swu * sx1;
        ag[t][0] += cg[0] * fg0; ag[t][1] += cg[1] * fg1; ag[t][2] += cg[2] * fg0; ag[t][3] += cg[3] * fg1;
        au[t][0] += cu[0] * fu0; au[t][1] += cu[1] * fu1; au[t][2] += cu[2] * fu0; au[t][3] += cu[3] * fu1;
      }
    }
    cp_async_wait<0>();
    __syncthreads();
    // cross-warp reduction over k: red[warp][row 0..31][token], rows 0..15 gate, 16..31 up
    float* red = reinterpret_cast<float*>(sm.ring);
    constexpr int kT = C::kTok;
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      const int tl = t * 8 + 2 * q;
      float* r = red + warp * 32 * kT;
      r[g * kT + tl] = ag[t][0];
      r[g * kT + tl + 1] = ag[t][1];
      r[(g + 8) * kT + tl] = ag[t][2];
      r[(g + 8) * kT + tl + 1] = ag[t][3];
      r[(16 + g) * kT + tl] = au[t][0];
      r[(16 + g) * kT + tl + 1] = au[t][1];
      r[(24 + g) * kT + tl] = au[t][2];
      r[(24 + g) * kT + tl + 1] = au[t][3];
    }
    __syncthreads();
    for (int idx = tid; idx < kSliceA * kT; idx += kThreads) {
      const int i = idx % kSliceA, tl = idx / kSliceA, n = p0 + tl;
      if (n < s.nt) {
        float gs = 0.f, us = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          gs += red[w * 32 * kT + i * kT + tl];
          us += red[w * 32 * kT + (16 + i) * kT + tl];
        }
        const float z = fminf(gs, p.limit);
        const float hv = z / (1.f + expf(-z)) * fminf(fmaxf(us, -p.limit), p.limit);
        p.h[(size_t)(s.hbase + n) * p.Imax + rg + i] = hv;
      }
    }
    __syncthreads();
  }

  // the 8th finished slice of a 128-column group quantises the group
  if (tid == 0) {
    __threadfence();
    const int old = atomicAdd(p.gcount + slot * p.gI + sl / (kBlock / kSliceA), 1);
    s_last = old == kBlock / kSliceA - 1;
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    const int grp = sl / (kBlock / kSliceA);
    for (int n = warp; n < s.nt; n += kWarps) {
      const size_t row = (size_t)(s.hbase + n);
      const float4 v = ld_l2f4(p.h + row * p.Imax + grp * kBlock + 4 * lane);
      const float amax = warp_max(fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
      const float sc = group_scale(amax, p.e8m0);
      *reinterpret_cast<uint32_t*>(p.hq + row * p.Imax + grp * kBlock + 4 * lane) =
          f32x4_to_e4m3x4(__fdiv_rn(v.x, sc), __fdiv_rn(v.y, sc), __fdiv_rn(v.z, sc), __fdiv_rn(v.w, sc));
      if (lane == 0) p.hs[row * p.gI + grp] = sc;
    }
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      if (!(fault && slot == 0)) atomicAdd(p.ready + slot, 1);
    }
  }
}

// ------------------------------------------------------------------ B item
template <int TT>
__device__ void run_B(const ExpertArgs& p, const Smem& sm, const Slot& s, int slot, int rb) {
  using C = Cfg<TT>;
  __shared__ int s_ok;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, q = lane & 3;
  const int nkb = s.Ie / kBlock;
  const int row0 = rb * kRowsB + warp * 16;
  const size_t Ie = s.Ie;
  const uint8_t* w0 = s.w2 + (size_t)(row0 + g) * Ie + 16 * q;
  const uint8_t* w1 = w0 + 8 * Ie;
  uint8_t* ring = sm.ring + warp * C::kRingWarp;

  if (tid == 0) {
    int ok = 1;
    if (ld_acquire(p.ready + slot) < nkb) {
      const unsigned long long t0 = globaltimer_ns();
      for (long it = 0;; ++it) {
        if (ld_acquire(p.ready + slot) >= nkb) break;
        if (*(volatile int*)(p.hdr + kHdrStatus) != 0 || it > (1l << 24)) { ok = 0; break; }
        if (globaltimer_ns() - t0 > kWaitNs) {
          atomicExch(p.hdr + kHdrStatus, MOE_ERR_DEVICE_TIMEOUT);
          ok = 0;
          break;
        }
        __nanosleep(128);
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  if (!s_ok) return;

  for (int p0 = 0; p0 < s.nt; p0 += C::kTok) {
    int hrow[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      const int n = p0 + t * 8 + g;
      hrow[t] = n < s.nt ? s.hbase + n : -1;
    }
    auto issue = [&](int kb, int st) {
      uint8_t* b = ring + st * C::kStage;
      const size_t ko = (size_t)kb * kBlock;
      cp_async16(b + (0 * 32 + lane) * 16, w0 + ko, true);
      cp_async16(b + (1 * 32 + lane) * 16, w0 + ko + 64, true);
      cp_async16(b + (2 * 32 + lane) * 16, w1 + ko, true);
      cp_async16(b + (3 * 32 + lane) * 16, w1 + ko + 64, true);
      uint8_t* xb = b + C::kStageW;
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const uint8_t* src = p.hq + (size_t)(hrow[t] < 0 ? 0 : hrow[t]) * p.Imax + ko + 16 * q;
        cp_async16(xb + ((2 * t) * 32 + lane) * 16, src, hrow[t] >= 0);
        cp_async16(xb + ((2 * t + 1) * 32 + lane) * 16, src + 64, hrow[t] >= 0);
      }
    };
#pragma unroll
    for (int i = 0; i < kNST - 1; ++i) {
      if (i < nkb) issue(i, i);
      cp_async_commit();
    }
    for (int idx = tid; idx < C::kTok * nkb; idx += kThreads) {
      const int n = p0 + idx / nkb, kb = idx % nkb;
      sm.sc[idx] = n < s.nt ? ld_l2f(p.hs + (size_t)(s.hbase + n) * p.gI + kb) : 0.f;
    }
    for (int kb = tid; kb < nkb; kb += kThreads)
      sm.sw[kb] = __ldg(s.s2 + (size_t)(rb * kRowsB / kBlock) * nkb + kb);
    __syncthreads();

    float acc[TT][4];
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
#pragma unroll 1
    for (int i = 0; i < nkb; ++i) {
      {
        const int j = i + kNST - 1;
        if (j < nkb) issue(j, j % kNST);
        cp_async_commit();
      }
      cp_async_wait<kNST - 1>();
      const uint4* b = reinterpret_cast<const uint4*>(ring + (i % kNST) * C::kStage);
      const uint4 a00 = b[0 * 32 + lane], a01 = b[1 * 32 + lane];
      const uint4 a10 = b[2 * 32 + lane], a11 = b[3 * 32 + lane];
      const float sw = sm.sw[i];
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const uint4 x0 = b[(8 + 2 * t) * 32 + lane], x1 = b[(9 + 2 * t) * 32 + lane];
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        mma_span_e4m3(c, a00, a10, x0);
        mma_span_e4m3(c, a01, a11, x1);
        const float f0 = sw * sm.sc[(t * 8 + 2 * q) * nkb + i], f1 = sw * sm.sc[(t * 8 + 2 * q + 1) * nkb + i];
        acc[t][0] += c[0] * f0; acc[t][1] += c[1] * f1; acc[t][2] += c[2] * f0; acc[t][3] += c[3] * f1;
      }
    }
    cp_async_wait<0>();
#pragma unroll
    for (int t = 0; t < TT; ++t) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int n = p0 + t * 8 + 2 * q + j;
        if (n < s.nt) {
          float* dst = s.shared ? p.shared_out + (size_t)n * p.H
                                : p.rows + (size_t)sm.sorted[s.o + n] * p.H;
          dst[row0 + g] = acc[t][j];
          dst[row0 + g + 8] = acc[t][2 + j];
        }
      }
    }
    __syncthreads();
  }
}

template <int TT>
__global__ void __launch_bounds__(kThreads) experts_kernel(ExpertArgs p) {
  using C = Cfg<TT>;
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int s_item;
  __shared__ int s_nact;
  const int tid = threadIdx.x;
  const int nkbMax = max(p.H, p.Imax) / kBlock;
  Smem sm;
  sm.ring = smem;
  sm.sc = reinterpret_cast<float*>(smem + C::kRing);
  sm.sw = sm.sc + C::kTok * nkbMax;
  sm.off = reinterpret_cast<int*>(sm.sw + 2 * nkbMax);
  sm.act = sm.off + (p.E + 1);
  sm.sorted = sm.act + p.E;

  if (tid == 0) {
    s_nact = *(volatile int*)(p.hdr + kHdrActive);
    s_item = atomicAdd(p.hdr + kHdrQueue, 1);
  }
  __syncthreads();
  const int n_act = s_nact;
  const int fault = *(volatile int*)(p.hdr + kHdrFault);
  for (int i = tid; i <= p.E; i += kThreads) sm.off[i] = p.off[i];
  for (int i = tid; i < n_act; i += kThreads) sm.act[i] = p.act[i];
  for (int i = tid; i < p.Mk; i += kThreads) sm.sorted[i] = p.sorted[i];
  __syncthreads();

  const bool has_shared = p.Is > 0;
  const int nA_sh = has_shared ? p.Is / kSliceA : 0;
  const int nA_r = p.I / kSliceA;
  const int nB = p.H / kRowsB;
  const int totA = nA_sh + n_act * nA_r;
  const int total = totA + ((has_shared ? 1 : 0) + n_act) * nB;

  int item = s_item;
  while (item < total) {
    __syncthreads();
    int nxt = 0;
    if (tid == 0) nxt = atomicAdd(p.hdr + kHdrQueue, 1);
    if (item < totA) {
      int slot, sl;
      if (item < nA_sh) { slot = 0; sl = item; }
      else { const int j = item - nA_sh; slot = j / nA_r + (has_shared ? 1 : 0); sl = j % nA_r; }
      const Slot s = make_slot(p, sm, slot, has_shared);
      run_A<TT>(p, sm, s, slot, sl, fault);
    } else {
      const int j = item - totA;
      const int slot = j / nB, rb = j % nB;
      const Slot s = make_slot(p, sm, slot, has_shared);
      run_B<TT>(p, sm, s, slot, rb);
    }
    if (tid == 0) s_item = nxt;
    __syncthreads();
    item = s_item;
  }
}

template <int TT>
size_t experts_smem(const ExpertArgs& a) {
  const int nkbMax = std::max(a.H, a.Imax) / kBlock;
  return Cfg<TT>::kRing + sizeof(float) * (Cfg<TT>::kTok * nkbMax + 2 * nkbMax) +
         sizeof(int) * (2 * a.E + 1 + a.Mk);
}

template <int TT>
cudaError_t launch_tt(const ExpertArgs& a, int num_sms, cudaStream_t s) {
  const size_t smem = experts_smem<TT>(a);
  cudaError_t err = cudaFuncSetAttribute(experts_kernel<TT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, experts_kernel<TT>, kThreads, smem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  experts_kernel<TT><<<per_sm * num_sms, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_experts(const ExpertArgs& a, int num_sms, cudaStream_t s) {
  if (a.M <= 8) return launch_tt<1>(a, num_sms, s);
  if (a.M <= 16) return launch_tt<2>(a, num_sms, s);
  return launch_tt<4>(a, num_sms, s);
}

}  // namespace moe
