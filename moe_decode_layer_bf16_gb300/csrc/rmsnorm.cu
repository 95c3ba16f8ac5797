// Layer boundary: weighted top-k finalize, residual add and RMSNorm.
//
// The draft page (vllm.models.glm5next.nvidia.specialized_decode.runtime.draft,
// SpecializedDraft.reduced_norm) makes the boundary return the normalised sum
// of the sublayer output and the residual, and the updated residual; on one
// GPU the tensor-parallel all-reduce it is fused with drops out.  The decode page (LayerStages._mega_moe) leaves the
// routed rows unfinalized in expanded order for this step, which weights them
// by the top-k weights and adds the shared expert.
//
// One token is spread over a cluster of 8 CTAs so that even a single-token
// step reads its (k+1) fp32 rows with 8 SMs; the 8 partial sums of squares
// are exchanged through distributed shared memory and added in rank order,
// so every CTA of the cluster computes the same (deterministic) norm.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace moe {

namespace {

constexpr int kCluster = 8;
constexpr int kThreads = 256;
constexpr int kMaxCols = 16384 / kCluster;
constexpr int kIter = kMaxCols / (kThreads * 4);  // 4-column groups a thread handles

// (two CTAs an SM: at 32 tokens the 256 CTAs then fit in one wave)
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 2)
    rmsnorm_kernel(NormArgs a) {
  __shared__ float s_rb[kMaxCols];
  __shared__ float s_warp[kThreads / 32];
  __shared__ float s_part;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int t = blockIdx.x / kCluster;
  const int ncol = a.H / kCluster, c0 = rank * ncol;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t rowo = (size_t)t * a.H + c0;
  const uint16_t* res = reinterpret_cast<const uint16_t*>(a.residual) + rowo;
  const uint16_t* xx = a.x ? reinterpret_cast<const uint16_t*>(a.x) + rowo : nullptr;
  const uint16_t* gain = reinterpret_cast<const uint16_t*>(a.gain) + c0;
  uint16_t* ro = reinterpret_cast<uint16_t*>(a.residual_out) + rowo;
  // The residual and the gain: inside the layer call (early) neither comes
  // from the kernels this one waits for, so they are loaded while those
  // finish; a stand-alone call loads them after the wait, like x.
  uint2 rv[kIter], gv[kIter];
  auto load_inputs = [&] {
#pragma unroll
    for (int i = 0; i < kIter; ++i) {
      const int j = tid * 4 + i * kThreads * 4;
      if (j < ncol) {
        rv[i] = *reinterpret_cast<const uint2*>(res + j);
        gv[i] = *reinterpret_cast<const uint2*>(gain + j);
      }
    }
  };
  const bool partial = a.m_out != nullptr;  // the same in every CTA
  if (a.early && !partial) load_inputs();
  grid_dep_wait();  // the rows come from the preceding expert kernel
  if (!a.early && !partial) load_inputs();

  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kIter; ++i) {
    const int j = tid * 4 + i * kThreads * 4;
    if (j >= ncol) break;
    float m[4] = {0.f, 0.f, 0.f, 0.f};
    if (xx) {
      const uint2 v = *reinterpret_cast<const uint2*>(xx + j);
      m[0] = bf16_lo(v.x); m[1] = bf16_hi(v.x); m[2] = bf16_lo(v.y); m[3] = bf16_hi(v.y);
    }
    if (a.rows) {
      // all k rows are loaded before any is added, so the loads overlap
      float w[kMaxTopK];
      float4 r[kMaxTopK];
#pragma unroll
      for (int s = 0; s < kMaxTopK; ++s) {
        if (s < a.k) {
          w[s] = a.route_w[(size_t)t * a.k + s];
          r[s] = *reinterpret_cast<const float4*>(a.rows + ((size_t)t * a.k + s) * a.H + c0 + j);
        }
      }
#pragma unroll
      for (int s = 0; s < kMaxTopK; ++s) {
        if (s < a.k) {
          m[0] += w[s] * r[s].x; m[1] += w[s] * r[s].y; m[2] += w[s] * r[s].z; m[3] += w[s] * r[s].w;
        }
      }
    }
    if (a.shared) {
      for (int pp = 0; pp < a.shared_parts; ++pp) {
        const float4 r = *reinterpret_cast<const float4*>(a.shared + (size_t)pp * a.M * a.H + rowo + j);
        m[0] += r.x; m[1] += r.y; m[2] += r.z; m[3] += r.w;
      }
    }
    if (partial) {  // a rank's partial sum of a tensor-parallel layer: fp32 m, nothing else
      *reinterpret_cast<float4*>(a.m_out + rowo + j) = make_float4(m[0], m[1], m[2], m[3]);
      continue;
    }
    const float r0 = m[0] + bf16_lo(rv[i].x), r1 = m[1] + bf16_hi(rv[i].x);
    const float r2 = m[2] + bf16_lo(rv[i].y), r3 = m[3] + bf16_hi(rv[i].y);
    const uint32_t p01 = pack_bf16(r0, r1), p23 = pack_bf16(r2, r3);
    *reinterpret_cast<uint2*>(ro + j) = make_uint2(p01, p23);
    const float b0 = bf16_lo(p01), b1 = bf16_hi(p01), b2 = bf16_lo(p23), b3 = bf16_hi(p23);
    s_rb[j] = b0; s_rb[j + 1] = b1; s_rb[j + 2] = b2; s_rb[j + 3] = b3;
    ss += b0 * b0 + b1 * b1 + b2 * b2 + b3 * b3;
  }
  if (partial) return;  // (uniform: no CTA of the cluster reaches its barriers)
  ss = warp_sum(ss);
  if (lane == 0) s_warp[warp] = ss;
  __syncthreads();
  if (tid == 0) {
    float v = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) v += s_warp[w];
    s_part = v;
  }
  cluster.sync();
  float total = 0.f;
  for (int r = 0; r < kCluster; ++r) total += *cluster.map_shared_rank(&s_part, r);
  cluster.sync();  // no CTA leaves while another still reads its s_part
  const float inv = 1.f / sqrtf(total / (float)a.H + a.eps);
  uint16_t* out = reinterpret_cast<uint16_t*>(a.out) + rowo;
#pragma unroll
  for (int i = 0; i < kIter; ++i) {
    const int j = tid * 4 + i * kThreads * 4;
    if (j >= ncol) break;
    const uint32_t p01 = pack_bf16(s_rb[j] * inv * bf16_lo(gv[i].x), s_rb[j + 1] * inv * bf16_hi(gv[i].x));
    const uint32_t p23 = pack_bf16(s_rb[j + 2] * inv * bf16_lo(gv[i].y), s_rb[j + 3] * inv * bf16_hi(gv[i].y));
    *reinterpret_cast<uint2*>(out + j) = make_uint2(p01, p23);
  }
}

}  // namespace

cudaError_t launch_rmsnorm(const NormArgs& a, cudaStream_t s) {
  if (a.M == 0) return cudaSuccess;
  PdlLaunch L(dim3(a.M * kCluster), dim3(kThreads), 0, s);
  return cudaLaunchKernelEx(&L.cfg, rmsnorm_kernel, a);
}

}  // namespace moe
