// Sparse attention forward over the top-k selected keys.
//
// ("Support Ring Attention with DeepSeek DSA Sparse Indexer", Forward Flow
// step 5: logits = where(mask, Q K^T * scale, -inf), softmax, P V. Here the
// mask is the selected list of each query intersected with causality, and
// no dense [S, S] mask exists.)
//
// One CTA per query row (b, t). The selected K/V rows of the query are
// gathered chunk by chunk (NK keys, 16-byte cp.async, double-buffered) into
// shared memory once and shared by all H heads: the heads are the MMA M
// dimension (16 per warp), so one gathered row feeds H dot products. The
// softmax runs online in fp32 (exp2 with scale*log2(e) folded in); O is written
// in bf16 and LSE (natural log) in fp32 for the backward pass.

#include "dsa_attn_common.cuh"

namespace dsa {
namespace {

template <int DQK, int DV, int NK, int NW>
__global__ void __launch_bounds__(NW * 32) attn_fwd_kernel(const AttnParams p) {
  using L = AttnLayout<DQK, DV, NK, NW>;
  constexpr int NT = NW * 32;
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* Q_s = reinterpret_cast<uint16_t*>(smem + L::kQ);
  uint16_t* K_s = reinterpret_cast<uint16_t*>(smem + L::kK);
  uint16_t* V_s = reinterpret_cast<uint16_t*>(smem + L::kV);
  int* idx_s = reinterpret_cast<int*>(smem + L::kIdx);
  int* meta = reinterpret_cast<int*>(smem + L::kMeta);

  const long long row = static_cast<long long>(gridDim.x) - 1 - blockIdx.x;
  const int b = static_cast<int>(row / p.S);
  const int t = static_cast<int>(row - static_cast<long long>(b) * p.S);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int kend = load_index_row(p, row, t, idx_s, meta, DSA_STAGE_FWD);
  // Q rows of this query (rows >= H are zero)
  for (int i = tid; i < NW * 16 * (DQK / 8); i += NT) {
    const int r = i / (DQK / 8), pc = i % (DQK / 8);
    const bool ok = r < p.H;
    const uint16_t* src = ok ? p.Q + (row * p.H + r) * DQK + pc * 8 : p.Q;
    cp_async_16(smem_u32(Q_s + r * L::KP + pc * 8), src, ok ? 16u : 0u);
  }
  const int nchunks = (kend + NK - 1) / NK;
  if (nchunks > 0) gather_kv<DQK, DV, NK, NT>(p, b, 0, kend, idx_s, K_s, V_s);
  cp_async_commit();

  float o[DV / 8][4];
#pragma unroll
  for (int n = 0; n < DV / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  uint32_t qf[DQK / 16][4];

#pragma unroll 1
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c & 1;
    if (c + 1 < nchunks)
      gather_kv<DQK, DV, NK, NT>(p, b, c + 1, kend, idx_s, K_s + (buf ^ 1) * NK * L::KP,
                                 V_s + (buf ^ 1) * NK * L::VP);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (c == 0) {
#pragma unroll
      for (int kk = 0; kk < DQK / 16; ++kk)
        ldsm_x4(qf[kk], smem_u32(Q_s + (warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * L::KP +
                                 kk * 16 + (lane >> 4) * 8));
    }
    const uint16_t* Kb = K_s + buf * NK * L::KP;
    const uint16_t* Vb = V_s + buf * NK * L::VP;

    // S = Q K^T for 16 heads x NK keys
    float sacc[NK / 8][4];
#pragma unroll
    for (int n = 0; n < NK / 8; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
#pragma unroll
    for (int np = 0; np < NK / 16; ++np) {
#pragma unroll
      for (int kk = 0; kk < DQK / 16; ++kk) {
        uint32_t bf[4];
        ldsm_x4(bf, smem_u32(Kb + (np * 16 + (lane & 7) + (lane >> 4) * 8) * L::KP + kk * 16 +
                             ((lane >> 3) & 1) * 8));
        mma_16816(sacc[2 * np], qf[kk], bf[0], bf[1]);
        mma_16816(sacc[2 * np + 1], qf[kk], bf[2], bf[3]);
      }
    }
    // mask + online softmax (rows lane/4 and lane/4 + 8 of this warp)
#pragma unroll
    for (int n = 0; n < NK / 8; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = c * NK + n * 8 + 2 * (lane & 3) + (e & 1);
        const bool valid = j < kend && idx_s[j] >= 0;
        sacc[n][e] = valid ? sacc[n][e] * p.scale_log2 : -INFINITY;
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float mx = mrow[r];
#pragma unroll
      for (int n = 0; n < NK / 8; ++n) mx = fmaxf(mx, fmaxf(sacc[n][2 * r], sacc[n][2 * r + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float base = mx == -INFINITY ? 0.f : mx;
      const float alpha = exp2f(mrow[r] - base);
      mrow[r] = mx;
      float ls = 0.f;
#pragma unroll
      for (int n = 0; n < NK / 8; ++n) {
        sacc[n][2 * r] = exp2f(sacc[n][2 * r] - base);
        sacc[n][2 * r + 1] = exp2f(sacc[n][2 * r + 1] - base);
        ls += sacc[n][2 * r] + sacc[n][2 * r + 1];
      }
      lrow[r] = lrow[r] * alpha + ls;
#pragma unroll
      for (int n = 0; n < DV / 8; ++n) {
        o[n][2 * r] *= alpha;
        o[n][2 * r + 1] *= alpha;
      }
    }
    // O += P V
#pragma unroll
    for (int k2 = 0; k2 < NK / 16; ++k2) {
      uint32_t a[4];
      a[0] = pack_bf16(sacc[2 * k2][0], sacc[2 * k2][1]);
      a[1] = pack_bf16(sacc[2 * k2][2], sacc[2 * k2][3]);
      a[2] = pack_bf16(sacc[2 * k2 + 1][0], sacc[2 * k2 + 1][1]);
      a[3] = pack_bf16(sacc[2 * k2 + 1][2], sacc[2 * k2 + 1][3]);
#pragma unroll
      for (int dp = 0; dp < DV / 16; ++dp) {
        uint32_t bf[4];
        ldsm_x4_t(bf, smem_u32(Vb + (k2 * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * L::VP +
                               dp * 16 + (lane >> 4) * 8));
        mma_16816(o[2 * dp], a, bf[0], bf[1]);
        mma_16816(o[2 * dp + 1], a, bf[2], bf[3]);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  // normalise and store
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float l = lrow[r];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    const int h = warp * 16 + (lane >> 2) + r * 8;
    if (h < p.H) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint32_t* orow = reinterpret_cast<uint32_t*>(p.O + (row * p.H + h) * DV);
#pragma unroll
      for (int n = 0; n < DV / 8; ++n)
        orow[(n * 8 + 2 * (lane & 3)) >> 1] = pack_bf16(o[n][2 * r] * inv, o[n][2 * r + 1] * inv);
      if ((lane & 3) == 0)
        p.lse[row * p.H + h] = l > 0.f ? (mrow[r] + log2f(l)) * 0.69314718055994530942f
                                       : -INFINITY;
    }
  }
}

template <int DQK, int DV, int NK, int NW>
int launch_fwd_t(const AttnParams& p, long long rows, cudaStream_t stream) {
  using L = AttnLayout<DQK, DV, NK, NW>;
  const size_t smem = L::bytes(p.k);
  auto kern = attn_fwd_kernel<DQK, DV, NK, NW>;
  if (smem > 227 * 1024) return DSA_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return DSA_ERR_CUDA;
  kern<<<static_cast<unsigned>(rows), NW * 32, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

template <int DQK, int DV>
int launch_fwd_dims(const AttnParams& p, long long rows, cudaStream_t stream) {
  const int nw = (p.H + 15) / 16;
  if (nw <= 1) return launch_fwd_t<DQK, DV, 32, 1>(p, rows, stream);
  if (nw <= 2) return launch_fwd_t<DQK, DV, 32, 2>(p, rows, stream);
  if (nw <= 4) return launch_fwd_t<DQK, DV, 64, 4>(p, rows, stream);
  return launch_fwd_t<DQK, DV, 64, 8>(p, rows, stream);
}

}  // namespace

int launch_attn_fwd(const void* Q, const void* K, const void* V, const int32_t* idx, int B, int S,
                    int H, int Dqk, int Dv, int k, float scale, void* O, float* lse,
                    cudaStream_t stream, int path, int Hkv, void* scratch) {
  AttnParams p = make_attn_params(Q, K, V, idx, B, S, H, k, scale);
  p.O = static_cast<uint16_t*>(O);
  p.lse = lse;
  p.Hkv = Hkv;
  p.scratch = static_cast<uint8_t*>(scratch);
  const long long rows = static_cast<long long>(B) * S;
  if (rows * H > 0x7fffffffLL || H > 128 || Hkv < 1 || H % Hkv != 0) return DSA_ERR_UNSUPPORTED;
  if (Hkv > 1 || path == kFwdPathDense)
    return attn_fwd_dense_supported(B, S, H, Dqk, Dv, scale) ? launch_attn_fwd_dense(p, Dqk, Dv, stream)
                                                             : DSA_ERR_UNSUPPORTED;
  const int kind = attn_fwd_kernel_kind(B, S, H, Dqk, Dv, k, scale);
  if (kind == kFwdDenseTc) return launch_attn_fwd_dense(p, Dqk, Dv, stream);
  if (kind == kFwdGatherTc) return launch_attn_fwd_tc(p, Dqk, Dv, stream);
  if (Dqk == 192 && Dv == 128) return launch_fwd_dims<192, 128>(p, rows, stream);
  if (Dqk == 128 && Dv == 128) return launch_fwd_dims<128, 128>(p, rows, stream);
  if (Dqk == 64 && Dv == 64) return launch_fwd_dims<64, 64>(p, rows, stream);
  if (Dqk == 32 && Dv == 32) return launch_fwd_dims<32, 32>(p, rows, stream);
  return DSA_ERR_UNSUPPORTED;
}

int attn_fwd_kernel_kind(int B, int S, int H, int Dqk, int Dv, int k, float scale, int Hkv) {
  if (Hkv > 1)
    return attn_fwd_dense_supported(B, S, H, Dqk, Dv, scale) ? kFwdDenseTc : -DSA_ERR_UNSUPPORTED;
  if (attn_fwd_dense_supported(B, S, H, Dqk, Dv, scale) && attn_fwd_dense_preferred(B, S, H, k))
    return kFwdDenseTc;
  if (attn_fwd_tc_supported(H, Dqk, Dv, scale)) return kFwdGatherTc;
  return kFwdMmaSync;
}

bool attn_dims_supported(int Dqk, int Dv) {
  return (Dqk == 192 && Dv == 128) || (Dqk == 128 && Dv == 128) || (Dqk == 64 && Dv == 64) ||
         (Dqk == 32 && Dv == 32);
}

}  // namespace dsa
