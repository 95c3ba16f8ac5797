// Skinny BF16 GEMMs streamed over the whole GPU (stream-K), used twice:
//  * splitk_gemm_bf16: Y = alpha * A . W^T, the split-K BF16 projection that
//    the vLLM specialized-decode draft page (module docstring;
//    SpecializedDraft.run, eh_proj) runs above two tokens;
//  * the MoE router: fp32 logits = x . W_gate^T (decode page,
//    LayerStages._router), fused with the activation FP8 quantisation, sigmoid
//    top-k, the routing weights and the stable route order (LayerStages
//    ._mega_moe: route_order, expanded_idx_to_permuted_idx).
//
// Design: the weight matrix is HBM-bound (2 bytes read per multiply-add per
// token tile), so the contraction runs on warp-level bf16 MMAs fed straight
// from 128-bit streaming loads, and the K dimension is divided over all CTAs
// so that every SM streams the same number of bytes.  A CTA owns a contiguous
// run of (token chunk, 64-row tile, k-block) cells; each run that covers part
// of a tile leaves one fp32 partial, and the last CTA to finish a tile sums
// the partials in segment order (deterministic) and applies the epilogue.
#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "../../include/moe_decode.h"

namespace moe {

namespace {

constexpr int kThreads = 128;  // 4 warps, 16 weight rows each: 64-row tiles

__device__ __forceinline__ int cta_of_cell(long long x, long long total, int G) {
  return (int)(((x + 1) * (long long)G + total - 1) / total) - 1;
}

struct Gemv {
  const uint8_t* A;  // bf16 [M, K] as bytes
  const uint8_t* W;  // bf16 [N, K]
  int M, N, K, nkb, n_tiles, n_chunks, G, max_segs;
  long long total;  // statically split cells
  float* partials;
  unsigned* tickets;  // one per (chunk, tile), then the tail's unit and exit counters
  int dyn_tiles, dyn_unit, dyn_nu;
};

// acc[tt] holds rows (g, g+8) x tokens (2q, 2q+1) of token tile tt for this
// warp's 16 rows, summed over k-blocks [kb0, kb1).
template <int TT>
__device__ __forceinline__ void gemv_segment_regs(const Gemv& d, int chunk, int tile, int kb0, int kb1,
                                             float (&acc)[TT][4]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
#pragma unroll
  for (int t = 0; t < TT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  const int row0 = tile * 64 + warp * 16;
  if (row0 >= d.N) return;
  const size_t rowb = (size_t)d.K * 2;
  const uint8_t* w0 = d.W + (size_t)(row0 + g) * rowb + q * 16;
  const uint8_t* w1 = w0 + 8 * rowb;
  const uint8_t* bp[TT];
  bool bv[TT];
#pragma unroll
  for (int t = 0; t < TT; ++t) {
    int n = chunk * 8 * TT + t * 8 + g;
    bv[t] = n < d.M;
    bp[t] = d.A + (size_t)(bv[t] ? n : 0) * rowb + q * 16;
  }
  // weights and activations of the next k-block are loaded before this one's MMAs
  uint4 c0[4], c1[4], b[TT][4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    c0[s] = ld_stream(w0 + (size_t)kb0 * 256 + s * 64);
    c1[s] = ld_stream(w1 + (size_t)kb0 * 256 + s * 64);
  }
#pragma unroll
  for (int t = 0; t < TT; ++t)
#pragma unroll
    for (int s = 0; s < 4; ++s)
      b[t][s] = bv[t] ? __ldg(reinterpret_cast<const uint4*>(bp[t] + (size_t)kb0 * 256 + s * 64))
                      : make_uint4(0, 0, 0, 0);
#pragma unroll 1
  for (int kb = kb0; kb < kb1; ++kb) {
    const bool more = kb + 1 < kb1;
    uint4 n0[4], n1[4], nb[TT][4];
    if (more) {
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        n0[s] = ld_stream(w0 + (size_t)(kb + 1) * 256 + s * 64);
        n1[s] = ld_stream(w1 + (size_t)(kb + 1) * 256 + s * 64);
      }
#pragma unroll
      for (int t = 0; t < TT; ++t)
#pragma unroll
        for (int s = 0; s < 4; ++s)
          nb[t][s] = bv[t] ? __ldg(reinterpret_cast<const uint4*>(bp[t] + (size_t)(kb + 1) * 256 + s * 64))
                           : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int t = 0; t < TT; ++t)
#pragma unroll
      for (int s = 0; s < 4; ++s) mma_span_bf16(acc[t], c0[s], c1[s], b[t][s]);
    if (more) {
#pragma unroll
      for (int s = 0; s < 4; ++s) { c0[s] = n0[s]; c1[s] = n1[s]; }
#pragma unroll
      for (int t = 0; t < TT; ++t)
#pragma unroll
        for (int s = 0; s < 4; ++s) b[t][s] = nb[t][s];
    }
  }
}

// Hands over the sums of segment seg (of nseg) of (chunk, tile) ct that this
// CTA computed: written out directly when the tile has one segment, else
// stored as partial sums; the CTA that stores a tile's last segment adds them
// all in segment order (deterministic) and writes the tile.  Called by all
// threads.
constexpr int kXPitch = 256 + 16;  // bytes a token row of a staged k-block (padded: no bank conflicts)

MOE_DEV void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
MOE_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
MOE_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// The same sums with the chunk's token rows staged in shared memory: the CTA
// copies each k-block's 8 TT rows once (cp.async, double-buffered, one
// barrier a k-block) and every warp reads its fragments from there, so that
// only the weights of two k-blocks stay in registers (at 16 and 32 tokens the
// register form holds the activations of two k-blocks too, which limits the
// CTAs an SM and hence the weight bytes in flight).  Called by all threads of
// the CTA.
template <int TT>
__device__ __forceinline__ void gemv_segment_smem(const Gemv& d, int chunk, int tile, int kb0, int kb1,
                                                  float (&acc)[TT][4]) {
  __shared__ __align__(16) uint8_t s_x[2][8 * TT][kXPitch];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
#pragma unroll
  for (int t = 0; t < TT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  const int row0 = tile * 64 + warp * 16;
  const bool rows = row0 < d.N;  // (a warp past N still stages and meets the barriers)
  const size_t rowb = (size_t)d.K * 2;
  const uint8_t* w0 = d.W + (size_t)(rows ? row0 + g : 0) * rowb + q * 16;
  const uint8_t* w1 = w0 + 8 * rowb;
  auto stage_x = [&](int kb, int buf) {
#pragma unroll
    for (int j = 0; j < TT; ++j) {
      const int idx = threadIdx.x + j * kThreads;  // 16-byte piece idx of the 8 TT x 256-byte block
      const int r = idx >> 4, c = idx & 15, n = chunk * 8 * TT + r;
      uint8_t* dst = &s_x[buf][r][c * 16];
      if (n < d.M) cp_async16(dst, d.A + (size_t)n * rowb + (size_t)kb * 256 + c * 16);
      else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
    cp_async_commit();
  };
  uint4 c0[4], c1[4];
  if (rows) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      c0[s] = ld_stream(w0 + (size_t)kb0 * 256 + s * 64);
      c1[s] = ld_stream(w1 + (size_t)kb0 * 256 + s * 64);
    }
  }
  stage_x(kb0, 0);
#pragma unroll 1
  for (int kb = kb0; kb < kb1; ++kb) {
    const int buf = (kb - kb0) & 1;
    const bool more = kb + 1 < kb1;
    uint4 n0[4], n1[4];
    if (more && rows) {
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        n0[s] = ld_stream(w0 + (size_t)(kb + 1) * 256 + s * 64);
        n1[s] = ld_stream(w1 + (size_t)(kb + 1) * 256 + s * 64);
      }
    }
    cp_async_wait_all();
    // every thread's copies of this k-block have landed, and every warp is
    // done with the other buffer (read in the previous k-block)
    __syncthreads();
    if (more) stage_x(kb + 1, buf ^ 1);
    if (rows) {
#pragma unroll
      for (int t = 0; t < TT; ++t)
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const uint4 b = *reinterpret_cast<const uint4*>(&s_x[buf][t * 8 + g][s * 64 + q * 16]);
          mma_span_bf16(acc[t], c0[s], c1[s], b);
        }
      if (more) {
#pragma unroll
        for (int s = 0; s < 4; ++s) { c0[s] = n0[s]; c1[s] = n1[s]; }
      }
    }
  }
  __syncthreads();  // (the buffers are rewritten by the next segment)
}

// kStage: the activations staged in shared memory (gemv_segment_smem), else
// held in registers (gemv_segment_regs; 8-token tiles only)
template <int TT, bool kStage>
__device__ __forceinline__ void gemv_segment(const Gemv& d, int chunk, int tile, int kb0, int kb1,
                                             float (&acc)[TT][4]) {
  static_assert(kStage || TT == 1, "wider tiles stage their activations");
  if constexpr (kStage) gemv_segment_smem<TT>(d, chunk, tile, kb0, kb1, acc);
  else gemv_segment_regs<TT>(d, chunk, tile, kb0, kb1, acc);
}

// Partial-sum slot of segment seg of (chunk, tile) ct: max_segs slots a
// statically split tile, then dyn_nu a tile of the dynamic tail.
__device__ __forceinline__ size_t part_slot(const Gemv& d, long long ct, int seg) {
  const long long ns = (long long)d.n_chunks * d.n_tiles - d.dyn_tiles;
  return (size_t)(ct < ns ? ct * d.max_segs : ns * d.max_segs + (ct - ns) * d.dyn_nu) + seg;
}

template <int TT, class Epi>
__device__ void finish_segment(const Gemv& d, long long ct, int seg, int nseg, const float (&acc)[TT][4], Epi epi) {
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  constexpr int kTileOut = 8 * TT * 64;
  const int chunk = (int)(ct / d.n_tiles), tile = (int)(ct % d.n_tiles);
  const int rl0 = warp * 16 + g, rl1 = rl0 + 8;
  if (nseg == 1) {
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      const int n0 = chunk * 8 * TT + t * 8 + 2 * q;
      const int r0 = tile * 64 + rl0, r1 = tile * 64 + rl1;
      if (r0 < d.N) {
        if (n0 < d.M) { epi(n0, r0, acc[t][0]); epi(n0, r1, acc[t][2]); }
        if (n0 + 1 < d.M) { epi(n0 + 1, r0, acc[t][1]); epi(n0 + 1, r1, acc[t][3]); }
      }
    }
    __syncthreads();
    return;
  }
  float* P = d.partials + part_slot(d, ct, seg) * kTileOut;
#pragma unroll
  for (int t = 0; t < TT; ++t) {
    const int tl0 = t * 8 + 2 * q;
    P[tl0 * 64 + rl0] = acc[t][0];
    P[(tl0 + 1) * 64 + rl0] = acc[t][1];
    P[tl0 * 64 + rl1] = acc[t][2];
    P[(tl0 + 1) * 64 + rl1] = acc[t][3];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // publishes this CTA's partial sums; the last segment's count also
    // acquires every other segment's (the barrier below passes it on)
    const unsigned old = atom_add_acq_rel(d.tickets + ct, 1u);
    s_last = (old == (unsigned)(nseg - 1));
  }
  __syncthreads();
  if (!s_last) return;
  const float* P0 = d.partials + part_slot(d, ct, 0) * kTileOut;
  // only the valid tokens of the chunk; the segment loads of one output are
  // independent and issued 16 at a time, then added in segment order
  const int ntok = min(8 * TT, d.M - chunk * 8 * TT);
  for (int idx = threadIdx.x; idx < ntok * 64; idx += kThreads) {
    const int tl = idx >> 6, rl = idx & 63;
    const int n = chunk * 8 * TT + tl, r = tile * 64 + rl;
    if (r < d.N) {
      float v = 0.f;
      for (int s = 0; s < nseg; s += 16) {
        float t[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) t[j] = s + j < nseg ? __ldcg(P0 + (size_t)(s + j) * kTileOut + idx) : 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) v += t[j];
      }
      epi(n, r, v);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) d.tickets[ct] = 0u;
}

// Runs this CTA's statically assigned cells.  epi(token, row, value)
// receives every finished output.
template <int TT, bool kStage, class Epi>
__device__ void gemv_streamk(const Gemv& d, Epi epi) {
  const int c = blockIdx.x;
  long long cur = (long long)c * d.total / d.G;
  const long long end = (long long)(c + 1) * d.total / d.G;
  while (cur < end) {
    const long long ct = cur / d.nkb;
    const int kb0 = (int)(cur % d.nkb);
    const int kb1 = (int)min((long long)d.nkb, kb0 + (end - cur));
    const int chunk = (int)(ct / d.n_tiles), tile = (int)(ct % d.n_tiles);
    const int first = cta_of_cell(ct * d.nkb, d.total, d.G);
    const int nseg = cta_of_cell(ct * d.nkb + d.nkb - 1, d.total, d.G) - first + 1;
    float acc[TT][4];
    gemv_segment<TT, kStage>(d, chunk, tile, kb0, kb1, acc);
    finish_segment<TT>(d, ct, c - first, nseg, acc, epi);
    cur += kb1 - kb0;
  }
}

// The dynamic tail: units of dyn_unit k-blocks of the last dyn_tiles (chunk,
// tile)s, taken one at a time from the unit counter; the last CTA to leave
// resets both tail counters for the next call.
template <int TT, bool kStage, class Epi>
__device__ void gemv_tail(const Gemv& d, Epi epi) {
  __shared__ int s_unit;
  const long long n_ct = (long long)d.n_chunks * d.n_tiles;
  const int units = d.dyn_tiles * d.dyn_nu;
  unsigned* next = d.tickets + n_ct;
  for (;;) {
    __syncthreads();  // (s_unit is rewritten below)
    if (threadIdx.x == 0) s_unit = (int)atomicAdd(next, 1u);
    __syncthreads();
    const int u = s_unit;
    if (u >= units) break;
    const long long ct = n_ct - d.dyn_tiles + u / d.dyn_nu;
    const int seg = u % d.dyn_nu;
    const int kb0 = seg * d.dyn_unit, kb1 = min(d.nkb, kb0 + d.dyn_unit);
    float acc[TT][4];
    gemv_segment<TT, kStage>(d, (int)(ct / d.n_tiles), (int)(ct % d.n_tiles), kb0, kb1, acc);
    finish_segment<TT>(d, ct, seg, d.dyn_nu, acc, epi);
  }
  // every CTA's last take came before its count here: the last one resets
  if (threadIdx.x == 0 && atom_add_acq_rel(d.tickets + n_ct + 1, 1u) == (unsigned)gridDim.x - 1) {
    d.tickets[n_ct] = 0u;
    d.tickets[n_ct + 1] = 0u;
  }
}

constexpr int kPdlCells = 4;  // cells a CTA prefetches into L2 before it waits (programmatic launch)

// (register budgets: 128 a thread at 8 and 16 tokens, 170 at 32, so that 4,
// 4 and 3 CTAs an SM keep their weight loads in flight, with the activations
// staged in shared memory)
template <int TT>
__global__ void __launch_bounds__(kThreads, TT == 1 ? 4 : TT == 2 ? 4 : 3) splitk_kernel(Gemv d, void* C, int c_fp32, float alpha, int pdl) {
  if (pdl) {
    // Launched while the kernel that writes A still runs: the weights of this
    // CTA's first cells go into L2 (a thread a 128-byte line), then the wait.
    const long long x0 = (long long)blockIdx.x * d.total / d.G;
    const long long x1 = min(x0 + kPdlCells, (long long)(blockIdx.x + 1) * d.total / d.G);
    for (long long x = x0; x < x1; ++x) {
      const int kb = (int)(x % d.nkb), tile = (int)((x / d.nkb) % d.n_tiles);
      const int row = tile * 64 + (threadIdx.x >> 1);
      if (row < d.N)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(d.W + (size_t)row * d.K * 2 + (size_t)kb * 256 +
                                                      (threadIdx.x & 1) * 128));
    }
    grid_dep_wait();
  }
  auto epi = [&](int n, int r, float v) {
    v *= alpha;
    if (c_fp32)
      reinterpret_cast<float*>(C)[(size_t)n * d.N + r] = v;
    else
      reinterpret_cast<__nv_bfloat16*>(C)[(size_t)n * d.N + r] = __float2bfloat16_rn(v);
  };
  // (staged activations at every width: measured faster for the projection,
  // the router's 8-token form keeps them in registers)
  gemv_streamk<TT, true>(d, epi);
  if (d.dyn_tiles > 0) gemv_tail<TT, true>(d, epi);
}

// ------------------------------------------------------------------ router

struct RouterDev {
  const float* bias;
  int E, k, e8m0, H;
  float scaling;
  float* logits;
  uint8_t* xq;
  float* xs;
  int* hdr;
  int* ids;
  float* tw;
  int* sorted;
  int* off;
  int* act;
  int* gcount;
  int n_gcount;
  int* ready;
  int n_ready;
  int32_t* user_ids;
  float* user_w;
  int32_t* user_sorted;
  int32_t* user_off;
};

// Maps a float (not NaN) onto an unsigned key with the same order.
__device__ __forceinline__ unsigned order_key(float v) {
  const unsigned u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Sigmoid top-k of one token by one warp: lane l holds experts l, l+32, ...
// Slots come out in descending selection value; an exact tie goes to the
// lower expert id.  Each slot is two warp reductions: the largest value key
// over the lanes' best remaining experts, then the smallest id among the
// lanes that hold it (measured: half the cycles of a shuffle arg-max).
// Lane j < k ends with slot j's id and unbiased score.
template <int kPer>
__device__ __forceinline__ void warp_topk(const RouterDev& r, const float* logit, int lane, int& my_id,
                                          float& my_s) {
  float sel[kPer], sc[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    if (e < r.E) {
      const float l = logit[e];
      const float s = 1.f / (1.f + expf(-l));
      sc[i] = s;
      const float v = r.bias ? s + r.bias[e] : s;
      sel[i] = v == v ? v : -INFINITY;  // a NaN never outranks a number
    } else {
      sc[i] = 0.f;
      sel[i] = -INFINITY;
    }
  }
  unsigned taken = 0;
  my_id = -1;
  my_s = 0.f;
  for (int j = 0; j < r.k; ++j) {
    // this lane's best remaining expert (the lower index wins a tie)
    int bi = -1;
    float bv = -INFINITY, bs = 0.f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      if (lane + 32 * i < r.E && !((taken >> i) & 1u) && (bi < 0 || sel[i] > bv)) {
        bv = sel[i]; bs = sc[i]; bi = i;
      }
    }
    const unsigned key = bi < 0 ? 0u : order_key(bv);
    const unsigned kmax = __reduce_max_sync(0xffffffffu, key);
    const int win = __reduce_min_sync(0xffffffffu, bi >= 0 && key == kmax ? lane + 32 * bi : 0x7fffffff);
    const float ws = __shfl_sync(0xffffffffu, bs, win & 31);
    if ((win & 31) == lane) taken |= 1u << (win >> 5);
    if (lane == j) { my_id = win; my_s = ws; }
  }
}

// CTAs that share the routing of the tokens (4 tokens a CTA: one a warp up to
// 256 tokens; measured 8 -> 64: M = 256 verify batch 1819 -> 1799 us, skewed
// M = 128 341 -> 331 us)
constexpr int kMaxFinish = 64;

// Top-k, routing weights and per-token outputs of the tokens of finisher f of
// F: warp w takes tokens 4 f + w, 4 f + w + 4 F, ...  Each warp stages its
// token's logits (written by other CTAs: read from L2) in shared memory.  A
// lone finisher (F = 1) also keeps the ids in shared memory (ids_sh) for the
// route order it builds next.
__device__ void route_tokens(const RouterDev& r, int M, int f, int F, int* ids_sh) {
  __shared__ __align__(16) float s_lg[kThreads / 32][kMaxExperts];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k = r.k, E = r.E;
  float* lg = s_lg[warp];
  for (int t = 4 * f + warp; t < M; t += 4 * F) {
    for (int i = lane * 4; i < E; i += 128)
      *reinterpret_cast<float4*>(lg + i) = __ldcg(reinterpret_cast<const float4*>(r.logits + (size_t)t * E + i));
    __syncwarp();
    int id;
    float s;
    if (E <= 256) warp_topk<8>(r, lg, lane, id, s);
    else warp_topk<kMaxExperts / 32>(r, lg, lane, id, s);
    const float sum = warp_sum(lane < k ? s : 0.f);
    if (lane < k) {
      const float w = s / sum * r.scaling;
      r.ids[t * k + lane] = id;
      if (ids_sh) ids_sh[t * k + lane] = id;
      r.tw[t * k + lane] = w;
      if (r.user_ids) r.user_ids[t * k + lane] = id;
      if (r.user_w) r.user_w[t * k + lane] = w;
    }
    __syncwarp();
  }
}

// Route order from all tokens' ids (written by the finishers, or already in
// s_ids when this CTA routed every token): histogram, exclusive scans, the
// list of active experts and the stable placement.
__device__ void route_order(const RouterDev& r, int M, int* s_ids, bool ids_in_smem) {
  __shared__ int s_cnt[kMaxExperts];
  __shared__ int s_cur[kMaxExperts];
  __shared__ int s_nact;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k = r.k, Mk = M * k, E = r.E;
  if (!ids_in_smem)
    for (int i = threadIdx.x; i < Mk; i += kThreads) s_ids[i] = __ldcg(r.ids + i);
  for (int e = threadIdx.x; e < E; e += kThreads) s_cnt[e] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < Mk; i += kThreads) atomicAdd(&s_cnt[s_ids[i]], 1);
  __syncthreads();
  if (warp == 0) {
    // exclusive scans of the counts and of the active flags
    const int per = (E + 31) / 32, b0 = lane * per;
    int cs = 0, as = 0;
    for (int e = b0; e < min(E, b0 + per); ++e) { cs += s_cnt[e]; as += s_cnt[e] > 0; }
    int ci = cs, ai = as;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int c2 = __shfl_up_sync(0xffffffffu, ci, o), a2 = __shfl_up_sync(0xffffffffu, ai, o);
      if (lane >= o) { ci += c2; ai += a2; }
    }
    int rc = ci - cs, ra = ai - as;
    for (int e = b0; e < min(E, b0 + per); ++e) {
      r.off[e] = rc;
      if (r.user_off) r.user_off[e] = rc;
      s_cur[e] = rc;
      if (s_cnt[e] > 0) r.act[ra++] = e;
      rc += s_cnt[e];
    }
    if (lane == 31) {
      r.off[E] = ci;
      if (r.user_off) r.user_off[E] = ci;
      s_nact = ai;
    }
    __syncwarp();
    // stable placement, 32 routes at a time, in route order
    for (int base = 0; base < Mk; base += 32) {
      const int i = base + lane;
      const int e = i < Mk ? s_ids[i] : -1 - lane;
      const unsigned grp = __match_any_sync(0xffffffffu, e);
      const int leader = __ffs(grp) - 1;
      const int rank = __popc(grp & ((1u << lane) - 1u));
      int pos = 0;
      if (lane == leader && i < Mk) {
        pos = s_cur[e];
        s_cur[e] = pos + __popc(grp);
      }
      pos = __shfl_sync(0xffffffffu, pos, leader);
      if (i < Mk) {
        r.sorted[pos + rank] = i;
        if (r.user_sorted) r.user_sorted[pos + rank] = i;
      }
      __syncwarp();
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    r.hdr[kHdrActive] = s_nact;
    // this kernel's counters, for the next call (every CTA has passed them)
    r.hdr[kHdrRouterTicket] = 0;
    r.hdr[kHdrRouterFin] = 0;
  }
}

template <int TT>
__global__ void __launch_bounds__(kThreads, TT == 1 ? 4 : TT == 2 ? 3 : 2) router_kernel(Gemv d, RouterDev r) {
  __shared__ int s_finish;
  __shared__ int s_ids[kMaxMk];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dep_launch();  // the expert kernel may be scheduled on SMs this grid leaves free
  // (1) FP8 quantisation of x, per token per 128-column group, and (CTA 0) the
  // reset of the expert kernel's counters: the expert kernel starts on the
  // shared expert, which needs nothing else, as soon as every CTA has done this
  {
    if (blockIdx.x == 0) {
      for (int i = threadIdx.x; i < r.n_gcount; i += kThreads) r.gcount[i] = 0;
      for (int i = threadIdx.x; i < r.n_ready; i += kThreads) r.ready[i] = 0;
      if (threadIdx.x == 0) {
        r.hdr[kHdrQueue] = 0;
        r.hdr[kHdrDoneA] = 0;
      }
    }
    const int nkbH = r.H / kBlock;
    const int nsl = (nkbH + 7) / 8;  // slices per token
    const uint16_t* x = reinterpret_cast<const uint16_t*>(d.A);
    if (d.M * nkbH <= (int)gridDim.x * (kThreads / 32)) {
      // a few tokens: one warp per 128-column group (lane l holds columns
      // [4 l, 4 l + 4)), taken from the grid's last CTA down, so that the
      // CTAs that quantise, and start their logits after it, lose little
      // (one warp per 1024 columns kept two CTAs about 3 us behind the
      // others at one token, and the routing waits for the last logits)
      const int gi = ((int)gridDim.x - 1 - (int)blockIdx.x) * (kThreads / 32) + warp;
      if (gi < d.M * nkbH) {
        const int t = gi / nkbH, c0 = (gi % nkbH) * kBlock + 4 * lane;
        const uint2 raw = __ldg(reinterpret_cast<const uint2*>(x + (size_t)t * r.H + c0));
        const float v0 = bf16_lo(raw.x), v1 = bf16_hi(raw.x), v2 = bf16_lo(raw.y), v3 = bf16_hi(raw.y);
        float amax = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float sc = group_scale(amax, r.e8m0);
        *reinterpret_cast<uint32_t*>(r.xq + (size_t)t * r.H + c0) =
            f32x4_to_e4m3x4(__fdiv_rn(v0, sc), __fdiv_rn(v1, sc), __fdiv_rn(v2, sc), __fdiv_rn(v3, sc));
        if (lane == 0) r.xs[(size_t)t * nkbH + gi % nkbH] = sc;
      }
    } else {
      // one warp per 1024-column slice of a token (8 groups): lane l holds
      // columns [32 l, 32 l + 32) of the slice, a group is 4 lanes
      for (int si = blockIdx.x * (kThreads / 32) + warp; si < d.M * nsl; si += gridDim.x * (kThreads / 32)) {
        const int t = si / nsl, c0 = (si % nsl) * 1024 + 32 * lane;
        const bool on = c0 < r.H;
        uint4 raw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          raw[j] = on ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * r.H + c0 + 8 * j)) : make_uint4(0, 0, 0, 0);
        float v[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[8 * j + 0] = bf16_lo(raw[j].x); v[8 * j + 1] = bf16_hi(raw[j].x);
          v[8 * j + 2] = bf16_lo(raw[j].y); v[8 * j + 3] = bf16_hi(raw[j].y);
          v[8 * j + 4] = bf16_lo(raw[j].z); v[8 * j + 5] = bf16_hi(raw[j].z);
          v[8 * j + 6] = bf16_lo(raw[j].w); v[8 * j + 7] = bf16_hi(raw[j].w);
        }
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        if (on) {
          const float sc = group_scale(amax, r.e8m0);
          uint32_t q[8];
#pragma unroll
          for (int j = 0; j < 8; ++j)
            q[j] = f32x4_to_e4m3x4(__fdiv_rn(v[4 * j], sc), __fdiv_rn(v[4 * j + 1], sc), __fdiv_rn(v[4 * j + 2], sc),
                                   __fdiv_rn(v[4 * j + 3], sc));
          uint8_t* dst = r.xq + (size_t)t * r.H + c0;
          *reinterpret_cast<uint4*>(dst) = make_uint4(q[0], q[1], q[2], q[3]);
          *reinterpret_cast<uint4*>(dst + 16) = make_uint4(q[4], q[5], q[6], q[7]);
          if ((lane & 3) == 0) r.xs[(size_t)t * nkbH + c0 / kBlock] = sc;
        }
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      atomicAdd(r.hdr + kHdrXReady, 1);
    }
  }
  // (2) logits
  auto epi = [&](int n, int row, float v) { r.logits[(size_t)n * r.E + row] = v; };
  gemv_streamk<TT, (TT > 1)>(d, epi);
  // (3) the last F CTAs to finish their logits route the tokens (one warp per
  // token), once every CTA's logits are in; the last of them (or the only one,
  // from its own shared memory) builds the route order.  Every CTA of this
  // grid is resident (it launches before the expert kernel can), so the wait
  // ends; it is bounded.
  const int F = min(min(kMaxFinish, (d.M + 3) / 4), (int)gridDim.x);
  __syncthreads();
  if (threadIdx.x == 0) {
    const int t = atom_add_acq_rel(r.hdr + kHdrRouterTicket, 1);
    s_finish = t >= (int)gridDim.x - F ? t - ((int)gridDim.x - F) : -1;
  }
  __syncthreads();
  if (s_finish < 0) return;
  if (threadIdx.x == 0) {
    const unsigned long long t0 = globaltimer_ns();
    for (long n = 0; ld_acquire(r.hdr + kHdrRouterTicket) < (int)gridDim.x; ++n) {
      if (n > (1l << 22) || globaltimer_ns() - t0 > 200ull * 1000 * 1000) {
        atomicExch(r.hdr + kHdrStatus, MOE_ERR_DEVICE_TIMEOUT);
        break;
      }
      __nanosleep(32);
    }
  }
  __syncthreads();
  route_tokens(r, d.M, s_finish, F, F == 1 ? s_ids : nullptr);
  __syncthreads();
  if (F > 1) {
    // the last finisher to be done orders the routes, from every finisher's ids
    if (threadIdx.x == 0) {
      s_finish = atom_add_acq_rel(r.hdr + kHdrRouterFin, 1) == F - 1;
    }
    __syncthreads();
    if (!s_finish) return;
    __threadfence();
  }
  route_order(r, d.M, s_ids, F == 1);
}

Gemv make_gemv(const GemvPlan& p, const void* A, const void* W, float* partials, unsigned* tickets) {
  Gemv d;
  d.A = reinterpret_cast<const uint8_t*>(A);
  d.W = reinterpret_cast<const uint8_t*>(W);
  d.M = p.M; d.N = p.N; d.K = p.K; d.nkb = p.nkb; d.n_tiles = p.n_tiles; d.n_chunks = p.n_chunks;
  d.G = p.G; d.max_segs = p.max_segs; d.total = p.total;
  d.partials = partials;
  d.tickets = tickets;
  d.dyn_tiles = p.dyn_tiles; d.dyn_unit = p.dyn_unit; d.dyn_nu = p.dyn_nu;
  return d;
}

}  // namespace

static int cta_of_cell_host(long long x, long long total, int G) {
  return (int)(((x + 1) * (long long)G + total - 1) / total) - 1;
}

void plan_gemv(GemvPlan& p, int M, int N, int K, int G, int dyn_tiles) {
  p.M = M; p.N = N; p.K = K;
  p.chunk_tokens = gemv_chunk_tokens(M);
  p.n_chunks = (M + p.chunk_tokens - 1) / p.chunk_tokens;
  p.n_tiles = (N + 63) / 64;
  p.nkb = K / kBlock;
  const long long n_ct = (long long)p.n_chunks * p.n_tiles;
  p.dyn_tiles = dyn_tiles;
  p.dyn_unit = dyn_tiles > 0 ? std::min(kDynUnit, p.nkb) : 0;
  p.dyn_nu = dyn_tiles > 0 ? (p.nkb + p.dyn_unit - 1) / p.dyn_unit : 0;
  p.total = (n_ct - dyn_tiles) * p.nkb;
  p.G = (int)std::min<long long>(G, p.total);
  p.max_segs = 1;
  for (long long ct = 0; ct < n_ct - dyn_tiles; ++ct) {
    const int a = cta_of_cell_host(ct * p.nkb, p.total, p.G);
    const int b = cta_of_cell_host(ct * p.nkb + p.nkb - 1, p.total, p.G);
    p.max_segs = std::max(p.max_segs, b - a + 1);
  }
}

size_t gemv_partials_bytes(const GemvPlan& p) {
  const size_t n_ct = (size_t)p.n_chunks * p.n_tiles;
  const size_t slots = (n_ct - p.dyn_tiles) * p.max_segs + (size_t)p.dyn_tiles * p.dyn_nu;
  return slots * p.chunk_tokens * 64 * sizeof(float);
}

int gemv_blocks_per_sm(int chunk_tokens, bool router) {
  // per device; host threads may race on a first call (both store the same value)
  static std::atomic<int> cache[64][2][3];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  const int i = chunk_tokens == 8 ? 0 : (chunk_tokens == 16 ? 1 : 2);
  std::atomic<int>& slot = cache[dev][router ? 1 : 0][i];
  int c = slot.load(std::memory_order_relaxed);
  if (!c) {
    int n = 0;
    cudaError_t e;
    if (router)
      e = i == 0 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, router_kernel<1>, kThreads, 0)
        : i == 1 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, router_kernel<2>, kThreads, 0)
                 : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, router_kernel<4>, kThreads, 0);
    else
      e = i == 0 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, splitk_kernel<1>, kThreads, 0)
        : i == 1 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, splitk_kernel<2>, kThreads, 0)
                 : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, splitk_kernel<4>, kThreads, 0);
    c = (e == cudaSuccess && n > 0) ? n : 1;
    slot.store(c, std::memory_order_relaxed);
  }
  return c;
}

cudaError_t launch_splitk(const GemvPlan& p, const SplitKArgs& a, cudaStream_t s) {
  Gemv d = make_gemv(p, a.A, a.W, a.partials, a.tickets);
  const int pdl = a.pdl ? 1 : 0;
  auto kernel = p.chunk_tokens == 8 ? splitk_kernel<1> : p.chunk_tokens == 16 ? splitk_kernel<2> : splitk_kernel<4>;
  if (a.pdl) {
    PdlLaunch L(dim3(p.G), dim3(kThreads), 0, s);
    return cudaLaunchKernelEx(&L.cfg, kernel, d, a.C, a.c_fp32, a.alpha, pdl);
  }
  kernel<<<p.G, kThreads, 0, s>>>(d, a.C, a.c_fp32, a.alpha, pdl);
  return cudaGetLastError();
}

cudaError_t launch_router(const GemvPlan& p, const RouterArgs& a, cudaStream_t s) {
  Gemv d = make_gemv(p, a.x, a.W, a.partials, a.tickets);
  RouterDev r;
  r.bias = a.bias; r.E = a.E; r.k = a.k; r.e8m0 = a.e8m0; r.H = p.K; r.scaling = a.scaling;
  r.logits = a.logits; r.xq = a.xq; r.xs = a.xs; r.hdr = a.hdr; r.ids = a.ids; r.tw = a.tw;
  r.sorted = a.sorted; r.off = a.off; r.act = a.act; r.gcount = a.gcount; r.n_gcount = a.n_gcount;
  r.ready = a.ready; r.n_ready = a.n_ready; r.user_ids = a.user_ids; r.user_w = a.user_w;
  r.user_sorted = a.user_sorted; r.user_off = a.user_off;
  switch (p.chunk_tokens) {
    case 8: router_kernel<1><<<p.G, kThreads, 0, s>>>(d, r); break;
    case 16: router_kernel<2><<<p.G, kThreads, 0, s>>>(d, r); break;
    default: router_kernel<4><<<p.G, kThreads, 0, s>>>(d, r); break;
  }
  return cudaGetLastError();
}

}  // namespace moe

// ------------------------------------------------------------------ no-allocation split-K
// splitk_gemm_bf16_noalloc keeps its partial sums and tile counters in this
// file-scope device array instead of a caller workspace.  In host code the
// array's name is only a host-side stand-in: its device address is looked up
// once per device with cudaGetSymbolAddress and passed to the kernel.
namespace {
constexpr size_t kNoallocTicketBytes = 64 * 1024;  // up to 16384 (chunk, tile) counters
static __device__ __align__(256) uint8_t g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch on the current device; the lookup runs on
// the first call per device (host threads racing on it store the same value).
int noalloc_base(uint8_t** out) {
  static std::atomic<uint8_t*> base[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  uint8_t* b = base[dev].load(std::memory_order_acquire);
  if (!b) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return MOE_ERR_CUDA;
    b = reinterpret_cast<uint8_t*>(ptr);
    base[dev].store(b, std::memory_order_release);
  }
  *out = b;
  return MOE_OK;
}
}  // namespace

extern "C" int splitk_gemm_bf16_noalloc(const void* A, const void* W, void* C, int c_fp32, int M, int N, int K,
                                        int split_k, float alpha, void* stream) {
  using namespace moe;
  // the same plan (grid, split, reduction order) as splitk_gemm_bf16
  GemvPlan plan;
  int rc = plan_splitk(plan, M, N, K, split_k);
  if (rc != MOE_OK) return rc;
  if (!A || !W || !C) return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)A & 15u) || ((uintptr_t)W & 15u)) return MOE_ERR_INVALID_ARG;
  const size_t tickets = splitk_ticket_bytes(plan);
  if (tickets > kNoallocTicketBytes || kNoallocTicketBytes + splitk_partial_bytes(plan) > MOE_NOALLOC_SCRATCH_BYTES)
    return MOE_ERR_SCRATCH_LIMIT;
  uint8_t* base = nullptr;
  if ((rc = noalloc_base(&base)) != MOE_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  // the counters must start at zero whatever an earlier call left behind
  if (cudaMemsetAsync(base, 0, tickets, s) != cudaSuccess) return MOE_ERR_CUDA;
  SplitKArgs a;
  a.A = A; a.W = W; a.C = C; a.c_fp32 = c_fp32 ? 1 : 0; a.alpha = alpha;
  a.tickets = reinterpret_cast<unsigned*>(base);
  a.partials = reinterpret_cast<float*>(base + kNoallocTicketBytes);
  return launch_splitk(plan, a, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" int moe_debug_fill_noalloc_scratch(int byte, void* stream) {
  uint8_t* base = nullptr;
  const int rc = noalloc_base(&base);
  if (rc != MOE_OK) return rc;
  return cudaMemsetAsync(base, byte & 0xff, MOE_NOALLOC_SCRATCH_BYTES, (cudaStream_t)stream) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
