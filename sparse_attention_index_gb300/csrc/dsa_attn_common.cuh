// Pieces shared by the sparse-attention forward and backward kernels: the
// parameter block, the per-query index-row staging and the K/V row gather.
#pragma once

#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {

struct AttnParams {
  const uint16_t *Q, *K, *V, *O_in, *dO;
  const int32_t* idx;
  const float* lse_in;
  int B, S, H, k;
  int Hkv;     // K / V heads: head h reads K / V head h / (H / Hkv)
  float scale, scale_log2;
  uint16_t* O;
  float* lse;
  uint16_t* dQ;
  float* ws;   // fp32 [B*S, Dqk + Dv] dK / dV accumulators
  uint8_t* scratch;   // the dense-tile kernels' part of the caller's workspace (or null)
  int* err;    // device error word
  int test_drop_arrive;   // failure-detection test only: see attn_fwd_tc.cu
};

inline AttnParams make_attn_params(const void* Q, const void* K, const void* V,
                                   const int32_t* idx, int B, int S, int H, int k, float scale) {
  AttnParams p = {};
  p.Q = static_cast<const uint16_t*>(Q);
  p.K = static_cast<const uint16_t*>(K);
  p.V = static_cast<const uint16_t*>(V);
  p.idx = idx;
  p.B = B;
  p.S = S;
  p.H = H;
  p.Hkv = 1;
  p.k = k;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.err = device_error_word();
  return p;
}

// tcgen05 forward (attn_fwd_tc.cu): used for H <= 128 heads, (Dqk, Dv) = (192, 128) or
// (128, 128), and a positive scale.
bool attn_fwd_tc_supported(int H, int Dqk, int Dv, float scale);
int launch_attn_fwd_tc(const AttnParams& p, int Dqk, int Dv, cudaStream_t stream);

// tcgen05 forward on dense 128 x 128 tiles with a selection bitmap (attn_fwd_dense.cu):
// one query row per TMEM lane, so few heads still fill the M = 128 tile.
bool attn_fwd_dense_supported(int B, int S, int H, int Dqk, int Dv, float scale);
bool attn_fwd_dense_preferred(int B, int S, int H, int k);
int launch_attn_fwd_dense(const AttnParams& p, int Dqk, int Dv, cudaStream_t stream);
// The selection bitmap of the dense-tile kernels (attn_fwd_dense.cu): bits [B*S, W4]
// (W4 = 4 * QT words per row, written up to each row's own query tile), tile flags
// any [B, QT, QT] (zeroed by the caller), QT = ceil(S / 128).
void launch_dense_mask(const int32_t* idx, int B, int S, int k, int W4, int QT, uint32_t* bits,
                       uint8_t* any, int* err, cudaStream_t stream);
// Dense-tile backward (attn_bwd_dense.cu): dQ written directly, dK / dV added into the
// zeroed fp32 workspace p.ws like the other backward kernels.
bool attn_bwd_dense_supported(int B, int S, int H, int Dqk, int Dv, float scale);
bool attn_bwd_dense_preferred(int B, int S, int H, int k);
int launch_attn_bwd_dense(const AttnParams& p, int Dqk, int Dv, cudaStream_t stream);

// tcgen05 backward (attn_bwd_tc.cu): H <= 128, Dqk = 192, Dv = 128, positive scale.
// The fp32 dK/dV accumulator p.ws must already be zero on the stream.
bool attn_bwd_tc_supported(int H, int Dqk, int Dv, float scale);
int launch_attn_bwd_tc(const AttnParams& p, cudaStream_t stream);

// Shared-memory layout of the forward kernel: Q rows, two K/V chunk buffers
// (rows padded by 16 bytes so ldmatrix row addresses hit distinct banks), a
// small header and the query's index row.
template <int DQK, int DV, int NK, int NW>
struct AttnLayout {
  static constexpr int KP = DQK + 8;   // element pitch of Q / K rows
  static constexpr int VP = DV + 8;    // element pitch of V rows
  static constexpr size_t kQ = 0;
  static constexpr size_t kK = kQ + static_cast<size_t>(NW) * 16 * KP * 2;
  static constexpr size_t kV = kK + 2ull * NK * KP * 2;
  static constexpr size_t kMeta = kV + 2ull * NK * VP * 2;
  static constexpr size_t kIdx = kMeta + 16;
  static size_t bytes(int k) { return kIdx + ((static_cast<size_t>(k) + 3) & ~3ull) * 4; }
};

// Stage the index row of query (row, t) in shared memory. Entries outside
// [-1, S) are reported and dropped; entries above the diagonal are dropped
// (causal mask). Returns kend = 1 + the last position holding a key (0: none).
__device__ __forceinline__ int load_index_row(const AttnParams& p, long long row, int t,
                                              int* idx_s, int* meta, int stage) {
  if (threadIdx.x == 0) meta[0] = 0;
  __syncthreads();
  int last = 0;
  for (int j = threadIdx.x; j < p.k; j += blockDim.x) {
    int s = __ldg(p.idx + row * p.k + j);
    if (s < -1 || s >= p.S) {
      report_error(p.err, stage | DSA_DEVERR_BAD_INDEX);
      s = -1;
    }
    if (s > t) s = -1;
    idx_s[j] = s;
    if (s >= 0) last = j + 1;
  }
  if (last) atomicMax(&meta[0], last);
  __syncthreads();
  return meta[0];
}

// Gather the K and V rows of chunk c (positions c*NK .. c*NK+NK-1 of the index
// row) with 16-byte cp.async; rows without a key are zero-filled.
template <int DQK, int DV, int NK, int NT>
__device__ __forceinline__ void gather_kv(const AttnParams& p, int b, int c, int kend,
                                          const int* idx_s, uint16_t* Kdst, uint16_t* Vdst) {
  constexpr int PK = DQK / 8, PV = DV / 8, PER = PK + PV;
  constexpr int KP = DQK + 8, VP = DV + 8;
  for (int i = threadIdx.x; i < NK * PER; i += NT) {
    const int r = i / PER, pc = i - r * PER;
    const int j = c * NK + r;
    const int s = j < kend ? idx_s[j] : -1;
    const bool ok = s >= 0;
    const long long kv = static_cast<long long>(b) * p.S + (ok ? s : 0);
    if (pc < PK)
      cp_async_16(smem_u32(Kdst + r * KP + pc * 8), p.K + kv * DQK + pc * 8, ok ? 16u : 0u);
    else
      cp_async_16(smem_u32(Vdst + r * VP + (pc - PK) * 8), p.V + kv * DV + (pc - PK) * 8,
                  ok ? 16u : 0u);
  }
}

}  // namespace dsa
