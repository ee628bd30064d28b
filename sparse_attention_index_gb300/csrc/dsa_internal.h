// Launchers behind the C ABI. Each validates nothing (dsa_api.cu does) and
// returns a dsa_status after enqueueing its kernels on `stream`.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dsa {

// Device address of the library's error word on the current device.
int* device_error_word();

// The streaming form of the fused indexer + top-k (dsa_index_topk_stream): a sampled
// indexer pass scores sample_tiles(nkb) evenly spaced 128-key tiles of the nkb tiles of each
// query group's causal range (a 16th of them, at least 8 and at most kSampleTiles; all of
// them when there are fewer), kSampleKeys slots per row.
constexpr int kSampleTiles = 32;
constexpr int kSampleKeys = kSampleTiles * 128;
__host__ __device__ inline int sample_tiles(int nkb) {
  int nt = nkb / 16;
  nt = nt < 8 ? 8 : (nt > kSampleTiles ? kSampleTiles : nt);
  return nkb < nt ? nkb : nt;
}
constexpr int kStreamMaxS = 131072;     // keys per row the finishing kernel's bitmaps hold
constexpr int kStreamWindowCap = 4096;  // window keys listed per row
// the m-th of the nt tiles sampled out of nkb (increasing in m; every tile when nt == nkb)
__host__ __device__ inline int sample_tile(int m, int nt, int nkb) {
  return nt == nkb ? m : static_cast<int>((static_cast<long long>(m) * nkb) / nt);
}

// fp8 != 0: q_idx / k_idx are e4m3 bytes and k_scale (fp32 [B, S] or nullptr) scales
// each key's score.
int launch_index_scores(const void* q_idx, const void* k_idx, const void* w, int w_is_bf16,
                        const int32_t* seg, int B, int S, int Hi, int Di, float* scores,
                        int64_t ld, cudaStream_t stream, int fp8, const float* k_scale);

// rows [t_lo, t_hi) of every batch row only, scores of row t at row t - t_lo of a buffer with
// rows_blk rows per batch (the query-block form of the fused indexer + top-k; t_lo a
// multiple of 256)
int launch_index_scores_rows(const void* q_idx, const void* k_idx, const void* w, int w_is_bf16,
                             const int32_t* seg, int B, int S, int Hi, int Di, float* scores,
                             int64_t ld, cudaStream_t stream, int fp8, const float* k_scale,
                             int t_lo, int t_hi, long long rows_blk, const int* gate = nullptr);

// vals non-null: each slot's score as well ([B, S, k], -inf at slots without a key)
int launch_topk(const float* scores, int64_t ld, const int32_t* seg, int B, int S, int k,
                int32_t* idx, int32_t* count, float* vals, cudaStream_t stream);
// gate non-null: the kernels do nothing unless *gate != 0 (read on the device)
int launch_topk_rows(const float* scores, int64_t ld, const int32_t* seg, int B, int S, int k,
                     int32_t* idx, int32_t* count, float* vals, cudaStream_t stream, int t_lo,
                     int t_hi, long long rows_blk, const int* gate = nullptr);

// Streaming form passes. sample: [B*S, kSampleKeys] scores (NaN: not a valid key) of the
// sampled tiles. thr: [B*S, 2] (U, L) per row; cnt: [B*S, 4] zeroed before the emit pass;
// above: [B*S, k]; win: [B*S, cw] (key index, score bits).
int launch_index_sample(const void* q_idx, const void* k_idx, const void* w, int w_is_bf16,
                        const int32_t* seg, int B, int S, int Hi, int Di, cudaStream_t stream,
                        int fp8, const float* k_scale, float* sample);
int launch_index_emit(const void* q_idx, const void* k_idx, const void* w, int w_is_bf16,
                      const int32_t* seg, int B, int S, int Hi, int Di, cudaStream_t stream,
                      int fp8, const float* k_scale, const float* thr, int* cnt, int32_t* above,
                      float* above_vals, int k, int2* win, int cw);
// per row: (U, L) from the sample (rows with t < k: every valid key selected, -inf)
int launch_stream_window(const float* sample, const int32_t* seg, int B, int S, int G, int k,
                         float* thr, cudaStream_t stream);
// per row: the selection from the above / window lists into idx (in place) and count; a
// row the lists cannot settle sets flags[t / block_rows] = 1 and writes nothing
// vals (k <= 2048): the selected scores by slot; the emit pass wrote those of the keys
// >= U beside their list entries (above_vals)
int launch_stream_finish(const int32_t* seg, int B, int S, int k, const int* cnt,
                         const int2* win, int cw, int32_t* idx, int32_t* count, float* vals,
                         int* flags, int block_rows, cudaStream_t stream);

// path: kFwdPathAuto (the cheaper of the gathered-key and dense-tile kernels) or
// kFwdPathDense (the dense-tile kernel, DSA_ERR_UNSUPPORTED where it does not apply)
constexpr int kFwdPathAuto = 0, kFwdPathDense = 1;
// the kernel the automatic path runs: gathered-key tcgen05 (1 launch), dense-tile
// tcgen05 (bitmap build + attention: 2 launches) or mma.sync (1 launch)
constexpr int kFwdGatherTc = 0, kFwdDenseTc = 1, kFwdMmaSync = 2;
// Hkv > 1 (per-head or grouped K / V) runs on the dense-tile kernels only: the others
// share one K / V row between all heads. Returns -DSA_ERR_UNSUPPORTED where no kernel applies.
int attn_fwd_kernel_kind(int B, int S, int H, int Dqk, int Dv, int k, float scale, int Hkv = 1);
// scratch: the dense-tile kernels' scratch (dense_scratch_layout without Delta) or nullptr
// when the caller guarantees the dense-tile kernel is not taken
int launch_attn_fwd(const void* Q, const void* K, const void* V, const int32_t* idx, int B, int S,
                    int H, int Dqk, int Dv, int k, float scale, void* O, float* lse,
                    cudaStream_t stream, int path, int Hkv, void* scratch);

// path: kBwdPathAuto (the cheaper of the gathered-key and dense-tile kernels),
// kBwdPathNoAlloc (never the dense-tile kernels, whose scratch lives in the caller's
// workspace) or kBwdPathDense (the dense-tile kernels, DSA_ERR_UNSUPPORTED where they
// do not apply)
constexpr int kBwdPathAuto = 0, kBwdPathNoAlloc = 1, kBwdPathDense = 2;
// the kernels the automatic path runs: gathered-key tcgen05 (+ finalize: 2 launches),
// dense-tile tcgen05 (bitmap, dq, dk/dv, finalize: 4) or mma.sync (+ finalize: 2)
constexpr int kBwdGatherTc = 0, kBwdDenseTc = 1, kBwdMmaSync = 2;
int attn_bwd_kernel_kind(int B, int S, int H, int Dqk, int Dv, int k, float scale, int Hkv = 1);
// ws_dkv: the fp32 dK / dV accumulators; scratch: the dense-tile kernels' scratch
// (dense_scratch_layout with Delta) or nullptr on kBwdPathNoAlloc
int launch_attn_bwd(const void* Q, const void* K, const void* V, const int32_t* idx,
                    const void* O, const float* lse, const void* dO, int B, int S, int H, int Dqk,
                    int Dv, int k, float scale, void* dQ, void* dK, void* dV, float* ws_dkv,
                    cudaStream_t stream, int path, int Hkv, void* scratch);

bool attn_dims_supported(int Dqk, int Dv);

// Host validation shared by the attention entry points (dsa_api.cu, attn_bwd_noalloc.cu):
// DSA_OK, DSA_ERR_INVALID_ARG (null or misaligned pointer, bad size) or DSA_ERR_UNSUPPORTED
// (H > 128, head dims without a kernel), in that order of precedence.
int attn_fwd_args_status(const void* Q, const void* K, const void* V, const int32_t* idx, int B,
                         int S, int H, int Hkv, int Dqk, int Dv, int k, const void* O,
                         const void* lse);
int attn_bwd_args_status(const void* Q, const void* K, const void* V, const int32_t* idx,
                         const void* O, const void* lse, const void* dO, int B, int S, int H,
                         int Hkv, int Dqk, int Dv, int k, const void* dQ, const void* dK,
                         const void* dV);

// Scratch of the dense-tile attention kernels, carved from the caller's workspace: the
// selection bitmap [B*S, 4*QT] uint32 (QT = ceil(S / 128) query tiles of 128 rows), the
// tile flags [B, QT, QT] bytes and, for the backward, Delta fp32 [B*S, H]; each part
// starts on a 256-byte boundary. bytes = 0 when the dense-tile kernels cannot take the
// shape (dense_tiles_fit false), so nothing is reserved for it.
struct DenseScratch {
  size_t bits_off, any_off, delta_off, bytes;
};
bool dense_tiles_fit(int S, int H, int Hkv, int Dqk, int Dv);
DenseScratch dense_scratch_layout(int B, int S, int H, int Hkv, int Dqk, int Dv, bool delta);
// the backward's workspace: fp32 dK / dV accumulators [B*S*Hkv, Dqk + Dv], then (from
// this offset, a multiple of 256) the dense-tile scratch
size_t bwd_accumulator_bytes(int B, int S, int Hkv, int Dqk, int Dv);

// indexer auxiliary loss: target, KL and dI (kl zeroed here), then the gradient into
// q_idx, k_idx and w (dk zeroed here)
bool indexer_loss_supported(int H, int Dqk, float scale);
bool indexer_loss_bwd_supported(int Hi, int Di);
int launch_indexer_loss(const void* Q, const void* K, const int32_t* idx, const float* lse,
                        const float* scores, int64_t ld, int B, int S, int H, int Dqk, int k,
                        float scale, float grad_scale, float* kl, float* dI,
                        cudaStream_t stream);
int launch_indexer_loss_bwd(const void* q_idx, const void* k_idx, const float* w,
                            const int32_t* idx, const float* dI, int B, int S, int Hi, int Di,
                            int k, float* dq, float* dk, float* dw, cudaStream_t stream);
// the same on the CUDA cores, for every other shape (iloss_simt.cu)
int launch_indexer_loss_simt(const void* Q, const void* K, const int32_t* idx, const float* lse,
                             const float* scores, int64_t ld, int B, int S, int H, int Hkv,
                             int Dqk, int k, float scale, float grad_scale, float* kl, float* dI,
                             cudaStream_t stream);
int launch_indexer_loss_bwd_simt(const void* q_idx, const void* k_idx, const float* w,
                                 const int32_t* idx, const float* dI, int B, int S, int Hi, int Di,
                                 int k, float* dq, float* dk, float* dw, cudaStream_t stream);
bool indexer_dims_supported(int Hi, int Di);

}  // namespace dsa
