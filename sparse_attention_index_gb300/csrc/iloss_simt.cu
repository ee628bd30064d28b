// The indexer's auxiliary loss for the shapes the tensor-core kernels (iloss.cu) do not
// take: any head count and head dims, and per-head or grouped K/V in the target. The
// same quantities as there ("Implement QK attention head chunking for CSA": the
// head-summed softmax target; "Support Ring Attention with DeepSeek DSA Sparse
// Indexer", Loss Harvesting & Objective Injection), on the CUDA cores: one CTA per query
// row, one warp per selected key.
//
//   target  pbar_j = (1/H) sum_h exp(scale Q[t,h].K[s_j, h / (H/Hkv)] - LSE[t,h])
//   student q_j = softmax_j(I[t, s_j]);  kl[t] = sum_j pbar_j (log pbar_j - log q_j)
//   dI_j = g (q_j - pbar_j)
//   dw[t,h] = sum_j dI_j max(0, z_hj);  dq[t,h] = sum_j dI_j w[t,h] [z_hj > 0] k[s_j]
//   dk[s_j] += sum_h dI_j w[t,h] [z_hj > 0] q[t,h]       (z_hj = q[t,h].k[s_j])

#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kSimtThreads = 256;
constexpr int kSimtWarps = kSimtThreads / 32;

__device__ __forceinline__ float bf16f(const __nv_bfloat16* p, long long i) {
  return __bfloat162float(p[i]);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// key in slot j of row (b, t) if selected (0 <= s <= t), else -1; out-of-range entries are
// reported and skipped
__device__ __forceinline__ int sel_key(const int32_t* irow, int j, int t, int S, int* err,
                                       int code) {
  const int s = irow[j];
  if (s < -1 || s >= S) {
    report_error(err, code);
    return -1;
  }
  return (s >= 0 && s <= t) ? s : -1;
}

struct SimtLossParams {
  const __nv_bfloat16 *Q, *K;
  const int32_t* idx;
  const float* lse;
  const float* scores;
  long long ld;
  int B, S, H, Hkv, Dqk, k;
  float scale, grad_scale;
  float* kl;
  float* dI;
  int* err;
};

__global__ void __launch_bounds__(kSimtThreads) loss_fwd_simt_kernel(const SimtLossParams p) {
  __shared__ float red_m[kSimtWarps], red_l[kSimtWarps], red_k[kSimtWarps];
  const long long row = blockIdx.x;
  const int t = static_cast<int>(row % p.S);
  const long long b = row / p.S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t* irow = p.idx + row * p.k;
  // the row's scores by key (ld > 0), or the selected keys' scores by slot (ld == 0)
  const float* srow = p.scores + row * (p.ld > 0 ? p.ld : p.k);
  auto score = [&](int s, int j) { return p.ld > 0 ? srow[s] : srow[j]; };
  const int code = DSA_STAGE_LOSS | DSA_DEVERR_BAD_INDEX;
  // log-sum-exp of the selected scores (the student's normaliser)
  float m = -INFINITY, l = 0.f;
  for (int j = tid; j < p.k; j += kSimtThreads) {
    const int s = sel_key(irow, j, t, p.S, p.err, code);
    if (s < 0) continue;
    const float v = score(s, j);
    if (v > m) {
      l = l * expf(m - v) + 1.f;
      m = v;
    } else if (v > -INFINITY) {
      l += expf(v - m);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, o), ol = __shfl_xor_sync(0xffffffffu, l, o);
    const float mm = fmaxf(m, om);
    l = (m > -INFINITY ? l * expf(m - mm) : 0.f) + (om > -INFINITY ? ol * expf(om - mm) : 0.f);
    m = mm;
  }
  if (lane == 0) {
    red_m[warp] = m;
    red_l[warp] = l;
  }
  __syncthreads();
  float M = -INFINITY, L = 0.f;
  for (int w2 = 0; w2 < kSimtWarps; ++w2) M = fmaxf(M, red_m[w2]);
  for (int w2 = 0; w2 < kSimtWarps; ++w2)
    if (red_m[w2] > -INFINITY) L += red_l[w2] * expf(red_m[w2] - M);
  const float logz = L > 0.f ? M + logf(L) : -INFINITY;
  // per selected key: the target over the heads (a lane per head), then dI and the loss
  const int grp = p.H / p.Hkv;
  float kl_acc = 0.f;
  for (int j = warp; j < p.k; j += kSimtWarps) {
    const int s = sel_key(irow, j, t, p.S, nullptr, 0);
    if (s < 0) {
      if (lane == 0) p.dI[row * p.k + j] = 0.f;
      continue;
    }
    float e = 0.f;
    for (int h = lane; h < p.H; h += 32) {
      const __nv_bfloat16* q = p.Q + (row * p.H + h) * p.Dqk;
      const __nv_bfloat16* kr = p.K + ((b * p.S + s) * p.Hkv + h / grp) * p.Dqk;
      float dot = 0.f;
      for (int d = 0; d < p.Dqk; ++d) dot = fmaf(bf16f(q, d), bf16f(kr, d), dot);
      e += expf(dot * p.scale - p.lse[row * p.H + h]);
    }
    e = warp_sum(e);
    if (lane == 0) {
      const float pbar = e / static_cast<float>(p.H);
      const float lq = score(s, j) - logz;
      p.dI[row * p.k + j] = p.grad_scale * (expf(lq) - pbar);
      if (pbar > 0.f) kl_acc += pbar * (logf(pbar) - lq);
    }
  }
  if (lane == 0) red_k[warp] = kl_acc;
  __syncthreads();
  if (tid == 0) {
    float kl = 0.f;
    for (int w2 = 0; w2 < kSimtWarps; ++w2) kl += red_k[w2];
    p.kl[row] = kl;
  }
}

struct SimtLossBwdParams {
  const __nv_bfloat16 *q, *kx;
  const float* w;
  const int32_t* idx;
  const float* dI;
  int B, S, Hi, Di, k;
  float *dq, *dk, *dw;   // dq and dw are written per row; dk is accumulated (zeroed first)
  int* err;
};

// one CTA per query row; dq_t [Hi x Di] and dw_t [Hi] accumulate in shared memory
__global__ void __launch_bounds__(kSimtThreads) loss_bwd_simt_kernel(const SimtLossBwdParams p) {
  extern __shared__ float acc[];   // dq [Hi * Di], then dw [Hi]
  const long long row = blockIdx.x;
  const int t = static_cast<int>(row % p.S);
  const long long b = row / p.S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nq = p.Hi * p.Di;
  for (int i = tid; i < nq + p.Hi; i += kSimtThreads) acc[i] = 0.f;
  __syncthreads();
  const int32_t* irow = p.idx + row * p.k;
  const __nv_bfloat16* qrow = p.q + row * p.Hi * p.Di;
  const float* wrow = p.w + row * p.Hi;
  const int code = DSA_STAGE_LOSS_BWD | DSA_DEVERR_BAD_INDEX;
  for (int j = warp; j < p.k; j += kSimtWarps) {
    const int s = sel_key(irow, j, t, p.S, p.err, code);
    if (s < 0) continue;
    const float g = p.dI[row * p.k + j];
    const __nv_bfloat16* kr = p.kx + (b * p.S + s) * p.Di;
    float* dkr = p.dk + (b * p.S + s) * p.Di;
    for (int h = 0; h < p.Hi; ++h) {
      // z = q[t,h] . k[s] across the lanes
      float z = 0.f;
      for (int d = lane; d < p.Di; d += 32) z = fmaf(bf16f(qrow, h * p.Di + d), bf16f(kr, d), z);
      z = warp_sum(z);
      if (!(z > 0.f)) continue;   // warp-uniform
      if (lane == 0) atomicAdd(&acc[nq + h], g * z);
      const float gw = g * wrow[h];
      for (int d = lane; d < p.Di; d += 32) {
        atomicAdd(&acc[h * p.Di + d], gw * bf16f(kr, d));
        atomicAdd(dkr + d, gw * bf16f(qrow, h * p.Di + d));
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < nq; i += kSimtThreads) p.dq[row * nq + i] = acc[i];
  for (int h = tid; h < p.Hi; h += kSimtThreads) p.dw[row * p.Hi + h] = acc[nq + h];
}

}  // namespace

int launch_indexer_loss_simt(const void* Q, const void* K, const int32_t* idx, const float* lse,
                             const float* scores, int64_t ld, int B, int S, int H, int Hkv,
                             int Dqk, int k, float scale, float grad_scale, float* kl, float* dI,
                             cudaStream_t stream) {
  SimtLossParams p;
  p.Q = static_cast<const __nv_bfloat16*>(Q);
  p.K = static_cast<const __nv_bfloat16*>(K);
  p.idx = idx;
  p.lse = lse;
  p.scores = scores;
  p.ld = ld;
  p.B = B;
  p.S = S;
  p.H = H;
  p.Hkv = Hkv;
  p.Dqk = Dqk;
  p.k = k;
  p.scale = scale;
  p.grad_scale = grad_scale;
  p.kl = kl;
  p.dI = dI;
  p.err = device_error_word();
  loss_fwd_simt_kernel<<<static_cast<unsigned>(static_cast<long long>(B) * S), kSimtThreads, 0,
                         stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

int launch_indexer_loss_bwd_simt(const void* q_idx, const void* k_idx, const float* w,
                                 const int32_t* idx, const float* dI, int B, int S, int Hi, int Di,
                                 int k, float* dq, float* dk, float* dw, cudaStream_t stream) {
  const size_t smem = (static_cast<size_t>(Hi) * Di + Hi) * sizeof(float);
  if (smem > 200 * 1024) return DSA_ERR_UNSUPPORTED;
  if (cudaMemsetAsync(dk, 0, sizeof(float) * static_cast<size_t>(B) * S * Di, stream) !=
      cudaSuccess)
    return DSA_ERR_CUDA;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(loss_bwd_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return DSA_ERR_CUDA;
  SimtLossBwdParams p;
  p.q = static_cast<const __nv_bfloat16*>(q_idx);
  p.kx = static_cast<const __nv_bfloat16*>(k_idx);
  p.w = w;
  p.idx = idx;
  p.dI = dI;
  p.B = B;
  p.S = S;
  p.Hi = Hi;
  p.Di = Di;
  p.k = k;
  p.dq = dq;
  p.dk = dk;
  p.dw = dw;
  p.err = device_error_word();
  loss_bwd_simt_kernel<<<static_cast<unsigned>(static_cast<long long>(B) * S), kSimtThreads,
                         smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
