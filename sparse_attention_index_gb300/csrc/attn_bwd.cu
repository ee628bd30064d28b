// Sparse attention backward over the top-k selected keys.
//
// ("Support Ring Attention with DeepSeek DSA Sparse Indexer", Backward Flow
// step 6: dQ = dP K, dK = dP^T Q, dV = P^T dO under the same mask, "dP" read
// as the gradient of the logits. The pages transpose their mask blocks to a
// key-major grid for dK / dV; here the query-major pass instead adds each
// selected key's partial dK / dV into an fp32 accumulator with vector atomics,
// which needs no transposed index.)
//
// One CTA per query row (b, t), 16 heads per warp:
//   prologue  Delta[h] = sum_c dO[t,h,c] O[t,h,c]   (the softmax-Jacobian term)
//   per chunk of NK selected keys (gathered K/V rows, double-buffered):
//     S  = Q K^T,  P = exp2(S*scale*log2e - lse*log2e)       (recomputed)
//     dP = dO V^T, dS = P (dP - Delta)
//     dQ += dS K                     (registers, whole row)
//     dK[s] += scale dS^T Q, dV[s] += P^T dO   (contraction over the heads
//                                               through shared memory, then
//                                               float2 atomics into ws)
//   epilogue  dQ * scale -> bf16
// A second small kernel turns the fp32 dK / dV accumulators into bf16.

#include "dsa_attn_common.cuh"

namespace dsa {
namespace {

template <int DQK, int DV, int NK, int NW>
struct BwdLayout {
  static constexpr int KP = DQK + 8, VP = DV + 8, PP = NK + 8;
  static constexpr int HR = NW * 16;   // head rows
  static constexpr size_t kQ = 0;
  static constexpr size_t kDO = kQ + static_cast<size_t>(HR) * KP * 2;
  static constexpr size_t kK = kDO + static_cast<size_t>(HR) * VP * 2;
  static constexpr size_t kV = kK + 2ull * NK * KP * 2;
  static constexpr size_t kP = kV + 2ull * NK * VP * 2;
  static constexpr size_t kDS = kP + static_cast<size_t>(HR) * PP * 2;
  static constexpr size_t kLse = kDS + static_cast<size_t>(HR) * PP * 2;
  static constexpr size_t kDelta = kLse + static_cast<size_t>(HR) * 4;
  static constexpr size_t kMeta = kDelta + static_cast<size_t>(HR) * 4;
  static constexpr size_t kIdx = kMeta + 16;
  static size_t bytes(int k) { return kIdx + ((static_cast<size_t>(k) + 3) & ~3ull) * 4; }
};

// C[NK keys x (2 x 8) cols] += A^T B over the head dimension, A stored
// [heads][keys] (pitch PP), B stored [heads][cols] (pitch BP); results go to
// the fp32 accumulator rows of the chunk's keys at column offset col0.
template <int NK, int NW, int NCOL, int PP, int BP>
__device__ __forceinline__ void head_contraction_atomic(const uint16_t* A_s, const uint16_t* B_s,
                                                        const int* key_of, int nkeys,
                                                        float* ws_base, int ws_pitch, int col0,
                                                        float mult) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int MT = NK / 16, NP = NCOL / 16, UNITS = MT * NP;
  for (int u = warp; u < UNITS; u += NW) {
    const int m = u % MT, np = u / MT;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int kh = 0; kh < NW; ++kh) {
      uint32_t a[4], bfr[4];
      ldsm_x4_t(a, smem_u32(A_s + (kh * 16 + (lane & 7) + (lane >> 4) * 8) * PP + m * 16 +
                            ((lane >> 3) & 1) * 8));
      ldsm_x4_t(bfr, smem_u32(B_s + (kh * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * BP +
                              np * 16 + (lane >> 4) * 8));
      mma_16816(acc[0], a, bfr[0], bfr[1]);
      mma_16816(acc[1], a, bfr[2], bfr[3]);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int kr = m * 16 + (lane >> 2) + r * 8;
      const int key = kr < nkeys ? key_of[kr] : -1;
      if (key < 0) continue;
      float* dst = ws_base + static_cast<long long>(key) * ws_pitch + col0;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int col = (2 * np + nt) * 8 + 2 * (lane & 3);
        atomicAdd(reinterpret_cast<float2*>(dst + col),
                  make_float2(acc[nt][2 * r] * mult, acc[nt][2 * r + 1] * mult));
      }
    }
  }
}

template <int DQK, int DV, int NK, int NW>
__global__ void __launch_bounds__(NW * 32) attn_bwd_kernel(const AttnParams p) {
  using L = BwdLayout<DQK, DV, NK, NW>;
  constexpr int NT = NW * 32;
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* Q_s = reinterpret_cast<uint16_t*>(smem + L::kQ);
  uint16_t* dO_s = reinterpret_cast<uint16_t*>(smem + L::kDO);
  uint16_t* K_s = reinterpret_cast<uint16_t*>(smem + L::kK);
  uint16_t* V_s = reinterpret_cast<uint16_t*>(smem + L::kV);
  uint16_t* P_s = reinterpret_cast<uint16_t*>(smem + L::kP);
  uint16_t* dS_s = reinterpret_cast<uint16_t*>(smem + L::kDS);
  float* lse_s = reinterpret_cast<float*>(smem + L::kLse);
  float* delta_s = reinterpret_cast<float*>(smem + L::kDelta);
  int* meta = reinterpret_cast<int*>(smem + L::kMeta);
  int* idx_s = reinterpret_cast<int*>(smem + L::kIdx);

  const long long row = static_cast<long long>(gridDim.x) - 1 - blockIdx.x;
  const int b = static_cast<int>(row / p.S);
  const int t = static_cast<int>(row - static_cast<long long>(b) * p.S);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q4 = lane & 3;

  const int kend = load_index_row(p, row, t, idx_s, meta, DSA_STAGE_BWD);
  for (int i = tid; i < L::HR * (DQK / 8); i += NT) {
    const int r = i / (DQK / 8), pc = i % (DQK / 8);
    const bool ok = r < p.H;
    cp_async_16(smem_u32(Q_s + r * L::KP + pc * 8), ok ? p.Q + (row * p.H + r) * DQK + pc * 8 : p.Q,
                ok ? 16u : 0u);
  }
  for (int i = tid; i < L::HR * (DV / 8); i += NT) {
    const int r = i / (DV / 8), pc = i % (DV / 8);
    const bool ok = r < p.H;
    cp_async_16(smem_u32(dO_s + r * L::VP + pc * 8),
                ok ? p.dO + (row * p.H + r) * DV + pc * 8 : p.dO, ok ? 16u : 0u);
  }
  const int nchunks = (kend + NK - 1) / NK;
  if (nchunks > 0) gather_kv<DQK, DV, NK, NT>(p, b, 0, kend, idx_s, K_s, V_s);
  cp_async_commit();

  // Delta and lse for this warp's heads (fp32, from the bf16 forward output)
  for (int hh = 0; hh < 16; ++hh) {
    const int h = warp * 16 + hh;
    float d = 0.f;
    if (h < p.H) {
      const uint16_t* orow = p.O_in + (row * p.H + h) * DV;
      const uint16_t* drow = p.dO + (row * p.H + h) * DV;
      for (int c = lane; c < DV; c += 32) d += bf16_bits_to_float(orow[c]) * bf16_bits_to_float(drow[c]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    if (lane == 0) {
      delta_s[h] = d;
      lse_s[h] = h < p.H ? p.lse_in[row * p.H + h] * 1.4426950408889634f : 0.f;
    }
  }

  float dq[DQK / 8][4];
#pragma unroll
  for (int n = 0; n < DQK / 8; ++n) dq[n][0] = dq[n][1] = dq[n][2] = dq[n][3] = 0.f;
  const int h0 = warp * 16 + g, h1 = h0 + 8;

#pragma unroll 1
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c & 1;
    if (c + 1 < nchunks)
      gather_kv<DQK, DV, NK, NT>(p, b, c + 1, kend, idx_s, K_s + (buf ^ 1) * NK * L::KP,
                                 V_s + (buf ^ 1) * NK * L::VP);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint16_t* Kb = K_s + buf * NK * L::KP;
    const uint16_t* Vb = V_s + buf * NK * L::VP;

    // S = Q K^T and dP = dO V^T for 16 heads x NK keys
    float s[NK / 8][4], dp[NK / 8][4];
#pragma unroll
    for (int n = 0; n < NK / 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[n][e] = dp[n][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < DQK / 16; ++kk) {
      uint32_t a[4];
      ldsm_x4(a, smem_u32(Q_s + (warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * L::KP +
                          kk * 16 + (lane >> 4) * 8));
#pragma unroll
      for (int np = 0; np < NK / 16; ++np) {
        uint32_t bf[4];
        ldsm_x4(bf, smem_u32(Kb + (np * 16 + (lane & 7) + (lane >> 4) * 8) * L::KP + kk * 16 +
                             ((lane >> 3) & 1) * 8));
        mma_16816(s[2 * np], a, bf[0], bf[1]);
        mma_16816(s[2 * np + 1], a, bf[2], bf[3]);
      }
    }
#pragma unroll
    for (int kk = 0; kk < DV / 16; ++kk) {
      uint32_t a[4];
      ldsm_x4(a, smem_u32(dO_s + (warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * L::VP +
                          kk * 16 + (lane >> 4) * 8));
#pragma unroll
      for (int np = 0; np < NK / 16; ++np) {
        uint32_t bf[4];
        ldsm_x4(bf, smem_u32(Vb + (np * 16 + (lane & 7) + (lane >> 4) * 8) * L::VP + kk * 16 +
                             ((lane >> 3) & 1) * 8));
        mma_16816(dp[2 * np], a, bf[0], bf[1]);
        mma_16816(dp[2 * np + 1], a, bf[2], bf[3]);
      }
    }
    // P and dS (registers), then to shared memory as bf16 [head][key]
    const float lse0 = lse_s[h0], lse1 = lse_s[h1];
    const float del0 = delta_s[h0], del1 = delta_s[h1];
    const bool hv0 = h0 < p.H, hv1 = h1 < p.H;
#pragma unroll
    for (int n = 0; n < NK / 8; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = c * NK + n * 8 + 2 * q4 + (e & 1);
        const bool hv = e < 2 ? hv0 : hv1;
        const bool valid = hv && j < kend && idx_s[j] >= 0;
        const float pr = valid ? exp2f(s[n][e] * p.scale_log2 - (e < 2 ? lse0 : lse1)) : 0.f;
        s[n][e] = pr;
        dp[n][e] = pr * (dp[n][e] - (e < 2 ? del0 : del1));
      }
      const int col = n * 8 + 2 * q4;
      *reinterpret_cast<uint32_t*>(P_s + (warp * 16 + g) * L::PP + col) = pack_bf16(s[n][0], s[n][1]);
      *reinterpret_cast<uint32_t*>(P_s + (warp * 16 + g + 8) * L::PP + col) =
          pack_bf16(s[n][2], s[n][3]);
      *reinterpret_cast<uint32_t*>(dS_s + (warp * 16 + g) * L::PP + col) =
          pack_bf16(dp[n][0], dp[n][1]);
      *reinterpret_cast<uint32_t*>(dS_s + (warp * 16 + g + 8) * L::PP + col) =
          pack_bf16(dp[n][2], dp[n][3]);
    }
    // dQ += dS K
#pragma unroll
    for (int k2 = 0; k2 < NK / 16; ++k2) {
      uint32_t a[4];
      a[0] = pack_bf16(dp[2 * k2][0], dp[2 * k2][1]);
      a[1] = pack_bf16(dp[2 * k2][2], dp[2 * k2][3]);
      a[2] = pack_bf16(dp[2 * k2 + 1][0], dp[2 * k2 + 1][1]);
      a[3] = pack_bf16(dp[2 * k2 + 1][2], dp[2 * k2 + 1][3]);
#pragma unroll
      for (int np = 0; np < DQK / 16; ++np) {
        uint32_t bf[4];
        ldsm_x4_t(bf, smem_u32(Kb + (k2 * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * L::KP +
                               np * 16 + (lane >> 4) * 8));
        mma_16816(dq[2 * np], a, bf[0], bf[1]);
        mma_16816(dq[2 * np + 1], a, bf[2], bf[3]);
      }
    }
    __syncthreads();
    // dK[s] += scale dS^T Q ; dV[s] += P^T dO   (contraction over all heads)
    const int* key_of = idx_s + c * NK;
    const int nkeys = kend - c * NK;   // positions past kend are never read
    float* ws_b = p.ws + static_cast<long long>(b) * p.S * (DQK + DV);
    head_contraction_atomic<NK, NW, DQK, L::PP, L::KP>(dS_s, Q_s, key_of, nkeys, ws_b, DQK + DV,
                                                       0, p.scale);
    head_contraction_atomic<NK, NW, DV, L::PP, L::VP>(P_s, dO_s, key_of, nkeys, ws_b, DQK + DV,
                                                      DQK, 1.f);
    __syncthreads();
  }
  cp_async_wait<0>();

  // dQ = scale * acc -> bf16
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int h = warp * 16 + g + r * 8;
    if (h < p.H) {
      uint32_t* drow = reinterpret_cast<uint32_t*>(p.dQ + (row * p.H + h) * DQK);
#pragma unroll
      for (int n = 0; n < DQK / 8; ++n)
        drow[(n * 8 + 2 * q4) >> 1] =
            pack_bf16(dq[n][2 * r] * p.scale, dq[n][2 * r + 1] * p.scale);
    }
  }
}

// fp32 [rows, Dqk + Dv] accumulators -> bf16 dK [rows, Dqk] and dV [rows, Dv]
__global__ void finalize_dkv_kernel(const float* __restrict__ ws, uint16_t* __restrict__ dK,
                                    uint16_t* __restrict__ dV, long long rows, int Dqk, int Dv) {
  const int D = Dqk + Dv;
  const long long n4 = rows * D / 4;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 v = reinterpret_cast<const float4*>(ws)[i];
    const long long e = i * 4;
    const long long r = e / D;
    const int c = static_cast<int>(e - r * D);
    uint2 packed;
    packed.x = pack_bf16(v.x, v.y);
    packed.y = pack_bf16(v.z, v.w);
    if (c < Dqk)
      *reinterpret_cast<uint2*>(dK + r * Dqk + c) = packed;
    else
      *reinterpret_cast<uint2*>(dV + r * Dv + (c - Dqk)) = packed;
  }
}

template <int DQK, int DV, int NK, int NW>
int launch_bwd_t(const AttnParams& p, long long rows, cudaStream_t stream) {
  using L = BwdLayout<DQK, DV, NK, NW>;
  const size_t smem = L::bytes(p.k);
  auto kern = attn_bwd_kernel<DQK, DV, NK, NW>;
  if (smem > 227 * 1024) return DSA_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return DSA_ERR_CUDA;
  kern<<<static_cast<unsigned>(rows), NW * 32, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

template <int DQK, int DV>
int launch_bwd_dims(const AttnParams& p, long long rows, cudaStream_t stream) {
  const int nw = (p.H + 15) / 16;
  if (nw <= 1) return launch_bwd_t<DQK, DV, 32, 1>(p, rows, stream);
  if (nw <= 2) return launch_bwd_t<DQK, DV, 32, 2>(p, rows, stream);
  if (nw <= 4) return launch_bwd_t<DQK, DV, 32, 4>(p, rows, stream);
  return launch_bwd_t<DQK, DV, 32, 8>(p, rows, stream);
}

}  // namespace

int attn_bwd_kernel_kind(int B, int S, int H, int Dqk, int Dv, int k, float scale, int Hkv) {
  if (Hkv > 1)
    return attn_bwd_dense_supported(B, S, H, Dqk, Dv, scale) ? kBwdDenseTc : -DSA_ERR_UNSUPPORTED;
  if (attn_bwd_dense_supported(B, S, H, Dqk, Dv, scale) && attn_bwd_dense_preferred(B, S, H, k))
    return kBwdDenseTc;
  if (attn_bwd_tc_supported(H, Dqk, Dv, scale)) return kBwdGatherTc;
  return kBwdMmaSync;
}

int launch_attn_bwd(const void* Q, const void* K, const void* V, const int32_t* idx,
                    const void* O, const float* lse, const void* dO, int B, int S, int H, int Dqk,
                    int Dv, int k, float scale, void* dQ, void* dK, void* dV, float* ws_dkv,
                    cudaStream_t stream, int path, int Hkv, void* scratch) {
  AttnParams p = make_attn_params(Q, K, V, idx, B, S, H, k, scale);
  p.Hkv = Hkv;
  p.O_in = static_cast<const uint16_t*>(O);
  p.lse_in = lse;
  p.dO = static_cast<const uint16_t*>(dO);
  p.dQ = static_cast<uint16_t*>(dQ);
  p.ws = ws_dkv;
  p.scratch = static_cast<uint8_t*>(scratch);
  const long long rows = static_cast<long long>(B) * S;
  if (rows * H > 0x7fffffffLL || H > 128 || Hkv < 1 || H % Hkv != 0) return DSA_ERR_UNSUPPORTED;
  const bool dense_ok = attn_bwd_dense_supported(B, S, H, Dqk, Dv, scale);
  // per-head or grouped K / V: the dense-tile kernels only, whose scratch the no-allocation
  // path does not have
  if (Hkv > 1 && (!dense_ok || path == kBwdPathNoAlloc)) return DSA_ERR_UNSUPPORTED;
  if (path == kBwdPathDense && !dense_ok) return DSA_ERR_UNSUPPORTED;
  if (cudaMemsetAsync(ws_dkv, 0, static_cast<size_t>(rows) * Hkv * (Dqk + Dv) * sizeof(float),
                      stream) != cudaSuccess)
    return DSA_ERR_CUDA;
  const bool dense = dense_ok && (Hkv > 1 || path == kBwdPathDense ||
                                  (path == kBwdPathAuto && attn_bwd_dense_preferred(B, S, H, k)));
  int rc;
  if (dense) rc = launch_attn_bwd_dense(p, Dqk, Dv, stream);
  else if (attn_bwd_tc_supported(H, Dqk, Dv, scale)) rc = launch_attn_bwd_tc(p, stream);
  else if (Dqk == 192 && Dv == 128) rc = launch_bwd_dims<192, 128>(p, rows, stream);
  else if (Dqk == 128 && Dv == 128) rc = launch_bwd_dims<128, 128>(p, rows, stream);
  else if (Dqk == 64 && Dv == 64) rc = launch_bwd_dims<64, 64>(p, rows, stream);
  else if (Dqk == 32 && Dv == 32) rc = launch_bwd_dims<32, 32>(p, rows, stream);
  else return DSA_ERR_UNSUPPORTED;
  if (rc != DSA_OK) return rc;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  finalize_dkv_kernel<<<sms * 4, 256, 0, stream>>>(ws_dkv, static_cast<uint16_t*>(dK),
                                                   static_cast<uint16_t*>(dV), rows * Hkv, Dqk,
                                                   Dv);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
