// The MTP layer's input: A[t] = [ enorm(E[id_t]) | hnorm(h_t) ] in bf16, the
// eh_proj projection's input ([draft page] vllm.models.glm5next.nvidia
// .specialized_decode.runtime.draft, SpecializedDraft.run: the embedding of
// the input tokens and the previous hidden state, each RMS-normalised with its
// own gain, then eh_proj).  The embedding half comes first.
//
// One CTA per token: both rows' sums of squares in one pass (fp32), one block
// reduction, then both normalised rows written.  The rows are re-read from L1
// in the second pass.  A token id outside [0, vocab) writes a zero embedding
// half and records MOE_ERR_INVALID_ARG in the status word (no read outside
// the table).
#include "common.cuh"
#include "kernels.h"
#include "../../include/moe_decode.h"

namespace moe {

namespace {

constexpr int kThreads = 512;

__global__ void __launch_bounds__(kThreads) eh_norm_kernel(EhNormArgs a) {
  __shared__ float s_red[2][kThreads / 32];
  grid_dep_launch();  // the projection may start streaming its weights now
  const int t = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int id = a.ids[t];
  const bool bad = id < 0 || id >= a.vocab;
  if (bad && tid == 0) atomicExch(a.status, MOE_ERR_INVALID_ARG);
  const uint16_t* e = bad ? nullptr : reinterpret_cast<const uint16_t*>(a.embed) + (size_t)id * a.H;
  const uint16_t* h = reinterpret_cast<const uint16_t*>(a.hidden) + (size_t)t * a.H;

  float se = 0.f, sh = 0.f;
  for (int j = tid * 4; j < a.H; j += kThreads * 4) {
    const uint2 hv = __ldg(reinterpret_cast<const uint2*>(h + j));
    const float h0 = bf16_lo(hv.x), h1 = bf16_hi(hv.x), h2 = bf16_lo(hv.y), h3 = bf16_hi(hv.y);
    sh += h0 * h0 + h1 * h1 + h2 * h2 + h3 * h3;
    if (e) {
      const uint2 ev = __ldg(reinterpret_cast<const uint2*>(e + j));
      const float e0 = bf16_lo(ev.x), e1 = bf16_hi(ev.x), e2 = bf16_lo(ev.y), e3 = bf16_hi(ev.y);
      se += e0 * e0 + e1 * e1 + e2 * e2 + e3 * e3;
    }
  }
  se = warp_sum(se);
  sh = warp_sum(sh);
  if (lane == 0) {
    s_red[0][warp] = se;
    s_red[1][warp] = sh;
  }
  __syncthreads();
  float te = 0.f, th = 0.f;
  for (int w = 0; w < kThreads / 32; ++w) {
    te += s_red[0][w];
    th += s_red[1][w];
  }
  const float inv_e = 1.f / sqrtf(te / (float)a.H + a.eps);
  const float inv_h = 1.f / sqrtf(th / (float)a.H + a.eps);

  const uint16_t* ge = reinterpret_cast<const uint16_t*>(a.enorm);
  const uint16_t* gh = reinterpret_cast<const uint16_t*>(a.hnorm);
  uint16_t* out = reinterpret_cast<uint16_t*>(a.out) + (size_t)t * 2 * a.H;
  for (int j = tid * 4; j < a.H; j += kThreads * 4) {
    uint2 re = make_uint2(0, 0);
    if (e) {
      const uint2 ev = __ldg(reinterpret_cast<const uint2*>(e + j));
      const uint2 gv = __ldg(reinterpret_cast<const uint2*>(ge + j));
      re = make_uint2(pack_bf16(bf16_lo(ev.x) * inv_e * bf16_lo(gv.x), bf16_hi(ev.x) * inv_e * bf16_hi(gv.x)),
                      pack_bf16(bf16_lo(ev.y) * inv_e * bf16_lo(gv.y), bf16_hi(ev.y) * inv_e * bf16_hi(gv.y)));
    }
    *reinterpret_cast<uint2*>(out + j) = re;
    const uint2 hv = __ldg(reinterpret_cast<const uint2*>(h + j));
    const uint2 gv = __ldg(reinterpret_cast<const uint2*>(gh + j));
    *reinterpret_cast<uint2*>(out + a.H + j) =
        make_uint2(pack_bf16(bf16_lo(hv.x) * inv_h * bf16_lo(gv.x), bf16_hi(hv.x) * inv_h * bf16_hi(gv.x)),
                   pack_bf16(bf16_lo(hv.y) * inv_h * bf16_lo(gv.y), bf16_hi(hv.y) * inv_h * bf16_hi(gv.y)));
  }
}

}  // namespace

cudaError_t launch_eh_norm(const EhNormArgs& a, cudaStream_t s) {
  if (a.M == 0) return cudaSuccess;
  eh_norm_kernel<<<a.M, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
