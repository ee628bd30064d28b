// The C ABI of libdsa.so: argument validation, then the kernel launchers.
// See include/dsa.h for the contract of every entry point.

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/dsa.h"
#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {

// The library's device error word (one per device that loads the library).
__device__ int g_device_error = 0;

int* device_error_word() {
  constexpr int kMaxDevices = 64;
  static int* addr[kMaxDevices] = {};
  static std::mutex lock;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  // host threads making their first call on a device at the same time fill one entry
  std::lock_guard<std::mutex> guard(lock);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<int*>(p);
  }
  return addr[dev];
}

}  // namespace dsa

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

namespace dsa {

int attn_fwd_args_status(const void* Q, const void* K, const void* V, const int32_t* idx, int B,
                         int S, int H, int Hkv, int Dqk, int Dv, int k, const void* O,
                         const void* lse) {
  if (!Q || !K || !V || !idx || !O || !lse) return DSA_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || H < 1 || Hkv < 1 || k < 1 || Dqk < 1 || Dv < 1)
    return DSA_ERR_INVALID_ARG;
  if (Dqk % 16 != 0 || Dv % 16 != 0 || H % Hkv != 0) return DSA_ERR_INVALID_ARG;
  const void* ptrs[] = {Q, K, V, idx, O, lse};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return DSA_ERR_INVALID_ARG;
  // Hkv > 1 runs on the dense-tile kernels only; the launchers refuse it elsewhere
  if (H > 128 || !attn_dims_supported(Dqk, Dv)) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

int attn_bwd_args_status(const void* Q, const void* K, const void* V, const int32_t* idx,
                         const void* O, const void* lse, const void* dO, int B, int S, int H,
                         int Hkv, int Dqk, int Dv, int k, const void* dQ, const void* dK,
                         const void* dV) {
  if (!dO || !dQ || !dK || !dV) return DSA_ERR_INVALID_ARG;
  const void* ptrs[] = {dO, dQ, dK, dV};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return DSA_ERR_INVALID_ARG;
  return attn_fwd_args_status(Q, K, V, idx, B, S, H, Hkv, Dqk, Dv, k, O, lse);
}

bool dense_tiles_fit(int S, int H, int Hkv, int Dqk, int Dv) {
  return S >= 1 && S <= 65536 && H >= 1 && H <= 128 && Hkv >= 1 && H % Hkv == 0 &&
         ((Dqk == 192 && Dv == 128) || (Dqk == 128 && Dv == 128));
}

namespace {
size_t round256(size_t n) { return (n + 255) / 256 * 256; }
}  // namespace

DenseScratch dense_scratch_layout(int B, int S, int H, int Hkv, int Dqk, int Dv, bool delta) {
  DenseScratch ly = {0, 0, 0, 0};
  if (B < 1 || !dense_tiles_fit(S, H, Hkv, Dqk, Dv)) return ly;
  const size_t QT = (static_cast<size_t>(S) + 127) / 128;
  const size_t rows = static_cast<size_t>(B) * S;
  ly.bits_off = 0;
  ly.any_off = round256(rows * QT * 4 * sizeof(uint32_t));
  ly.delta_off = round256(ly.any_off + static_cast<size_t>(B) * QT * QT);
  ly.bytes = delta ? round256(ly.delta_off + rows * H * sizeof(float)) : ly.delta_off;
  return ly;
}

size_t bwd_accumulator_bytes(int B, int S, int Hkv, int Dqk, int Dv) {
  if (B < 1 || S < 1 || Hkv < 1 || Dqk < 1 || Dv < 1) return 0;
  return round256(static_cast<size_t>(B) * S * Hkv * (Dqk + Dv) * sizeof(float));
}

}  // namespace dsa

extern "C" {

const char* dsa_status_string(int status) {
  switch (status) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT";
    case DSA_ERR_DEVICE: return "DSA_ERR_DEVICE";
    default: return "DSA_ERR_UNKNOWN";
  }
}

int dsa_version(void) { return 100; }

int dsa_get_last_device_error(void* stream, int32_t* code) {
  if (!code) return DSA_ERR_INVALID_ARG;
  *code = 0;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return DSA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, dsa::g_device_error, sizeof(int)) != cudaSuccess)
    return DSA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(dsa::g_device_error, &zero, sizeof(int)) != cudaSuccess)
      return DSA_ERR_CUDA;
  }
  *code = v;
  return DSA_OK;
}

int dsa_index_scores(const void* q_idx, const void* k_idx, const void* w, int w_dtype,
                     const int32_t* seg, int B, int S, int Hi, int Di, float* scores,
                     int64_t ld_scores, void* stream) {
  if (!q_idx || !k_idx || !w || !scores) return DSA_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || Hi < 1 || Di < 1) return DSA_ERR_INVALID_ARG;
  if (w_dtype != DSA_F32 && w_dtype != DSA_BF16) return DSA_ERR_INVALID_ARG;
  if (ld_scores < S || ld_scores % 4 != 0) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(w) || !aligned16(scores) ||
      (seg && !aligned16(seg)))
    return DSA_ERR_INVALID_ARG;
  if (Di % 8 != 0) return DSA_ERR_INVALID_ARG;
  if (!dsa::indexer_dims_supported(Hi, Di)) return DSA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * S * Hi >= (1LL << 31)) return DSA_ERR_UNSUPPORTED;
  return dsa::launch_index_scores(q_idx, k_idx, w, w_dtype == DSA_BF16, seg, B, S, Hi, Di,
                                  scores, ld_scores, as_stream(stream), 0, nullptr);
}

int dsa_index_scores_fp8(const void* q_idx, const void* k_idx, const float* k_scale,
                         const void* w, int w_dtype, const int32_t* seg, int B, int S, int Hi,
                         int Di, float* scores, int64_t ld_scores, void* stream) {
  if (!q_idx || !k_idx || !w || !scores) return DSA_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || Hi < 1 || Di < 1) return DSA_ERR_INVALID_ARG;
  if (w_dtype != DSA_F32 && w_dtype != DSA_BF16) return DSA_ERR_INVALID_ARG;
  if (ld_scores < S || ld_scores % 4 != 0) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(w) || !aligned16(scores) ||
      (seg && !aligned16(seg)) || (k_scale && !aligned16(k_scale)))
    return DSA_ERR_INVALID_ARG;
  if (Di % 16 != 0) return DSA_ERR_INVALID_ARG;
  if (!dsa::indexer_dims_supported(Hi, Di)) return DSA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * S * Hi >= (1LL << 31)) return DSA_ERR_UNSUPPORTED;
  return dsa::launch_index_scores(q_idx, k_idx, w, w_dtype == DSA_BF16, seg, B, S, Hi, Di,
                                  scores, ld_scores, as_stream(stream), 1, k_scale);
}

size_t dsa_topk_workspace_size(int B, int S, int k) {
  (void)B;
  (void)S;
  (void)k;
  return 0;
}

int dsa_topk(const float* scores, int64_t ld_scores, const int32_t* seg, int B, int S, int k,
             int32_t* idx, int32_t* count, float* vals, void* ws, size_t ws_bytes,
             void* stream) {
  (void)ws;
  (void)ws_bytes;
  if (!scores || !idx) return DSA_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || k < 1) return DSA_ERR_INVALID_ARG;
  if (ld_scores < S || ld_scores % 4 != 0) return DSA_ERR_INVALID_ARG;
  if (!aligned16(scores) || !aligned16(idx) || (seg && !aligned16(seg)) ||
      (count && !aligned16(count)) || (vals && !aligned16(vals)))
    return DSA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * S >= (1LL << 31)) return DSA_ERR_UNSUPPORTED;
  return dsa::launch_topk(scores, ld_scores, seg, B, S, k, idx, count, vals, as_stream(stream));
}

size_t dsa_sparse_attn_fwd_workspace_size(int B, int S, int H, int Hkv, int Dqk, int Dv) {
  return dsa::dense_scratch_layout(B, S, H, Hkv, Dqk, Dv, false).bytes;
}

}  // extern "C"

namespace {

int attn_fwd_impl(const void* Q, const void* K, const void* V, const int32_t* idx, int B, int S,
                  int H, int Hkv, int Dqk, int Dv, int k, float scale, void* O, float* lse,
                  void* ws, size_t ws_bytes, void* stream, int path) {
  const int rc = dsa::attn_fwd_args_status(Q, K, V, idx, B, S, H, Hkv, Dqk, Dv, k, O, lse);
  if (rc != DSA_OK) return rc;
  const size_t need = dsa_sparse_attn_fwd_workspace_size(B, S, H, Hkv, Dqk, Dv);
  if (need > 0 && (!ws || ws_bytes < need || !aligned16(ws))) return DSA_ERR_WORKSPACE;
  return dsa::launch_attn_fwd(Q, K, V, idx, B, S, H, Dqk, Dv, k, scale, O, lse,
                              as_stream(stream), path, Hkv, need > 0 ? ws : nullptr);
}

int attn_bwd_impl(const void* Q, const void* K, const void* V, const int32_t* idx, const void* O,
                  const float* lse, const void* dO, int B, int S, int H, int Hkv, int Dqk, int Dv,
                  int k, float scale, void* dQ, void* dK, void* dV, void* ws, size_t ws_bytes,
                  void* stream, int path) {
  const int rc = dsa::attn_bwd_args_status(Q, K, V, idx, O, lse, dO, B, S, H, Hkv, Dqk, Dv, k,
                                           dQ, dK, dV);
  if (rc != DSA_OK) return rc;
  const size_t need = dsa_sparse_attn_bwd_workspace_size(B, S, H, Hkv, Dqk, Dv);
  if (!ws || ws_bytes < need || !aligned16(ws)) return DSA_ERR_WORKSPACE;
  const size_t acc = dsa::bwd_accumulator_bytes(B, S, Hkv, Dqk, Dv);
  uint8_t* base = static_cast<uint8_t*>(ws);
  return dsa::launch_attn_bwd(Q, K, V, idx, O, lse, dO, B, S, H, Dqk, Dv, k, scale, dQ, dK, dV,
                              reinterpret_cast<float*>(base), as_stream(stream), path, Hkv,
                              need > acc ? base + acc : nullptr);
}

}  // namespace

extern "C" {

int dsa_sparse_attn_fwd(const void* Q, const void* K, const void* V, const int32_t* idx, int B,
                        int S, int H, int Hkv, int Dqk, int Dv, int k, float scale, void* O,
                        float* lse, void* ws, size_t ws_bytes, void* stream) {
  return attn_fwd_impl(Q, K, V, idx, B, S, H, Hkv, Dqk, Dv, k, scale, O, lse, ws, ws_bytes,
                       stream, dsa::kFwdPathAuto);
}

int dsa_sparse_attn_fwd_kernel(int B, int S, int H, int Hkv, int Dqk, int Dv, int k,
                               float scale) {
  if (B < 1 || S < 1 || H < 1 || k < 1) return -DSA_ERR_INVALID_ARG;
  if (Hkv < 1 || H % Hkv != 0) return -DSA_ERR_INVALID_ARG;
  if (H > 128 || !dsa::attn_dims_supported(Dqk, Dv)) return -DSA_ERR_UNSUPPORTED;
  return dsa::attn_fwd_kernel_kind(B, S, H, Dqk, Dv, k, scale, Hkv);
}

int dsa_sparse_attn_fwd_dense(const void* Q, const void* K, const void* V, const int32_t* idx,
                              int B, int S, int H, int Hkv, int Dqk, int Dv, int k, float scale,
                              void* O, float* lse, void* ws, size_t ws_bytes, void* stream) {
  return attn_fwd_impl(Q, K, V, idx, B, S, H, Hkv, Dqk, Dv, k, scale, O, lse, ws, ws_bytes,
                       stream, dsa::kFwdPathDense);
}

size_t dsa_sparse_attn_bwd_workspace_size(int B, int S, int H, int Hkv, int Dqk, int Dv) {
  const size_t acc = dsa::bwd_accumulator_bytes(B, S, Hkv, Dqk, Dv);
  if (acc == 0) return 0;
  return acc + dsa::dense_scratch_layout(B, S, H, Hkv, Dqk, Dv, true).bytes;
}

int dsa_sparse_attn_bwd(const void* Q, const void* K, const void* V, const int32_t* idx,
                        const void* O, const float* lse, const void* dO, int B, int S, int H,
                        int Hkv, int Dqk, int Dv, int k, float scale, void* dQ, void* dK, void* dV,
                        void* ws, size_t ws_bytes, void* stream) {
  return attn_bwd_impl(Q, K, V, idx, O, lse, dO, B, S, H, Hkv, Dqk, Dv, k, scale, dQ, dK, dV, ws,
                       ws_bytes, stream, dsa::kBwdPathAuto);
}

int dsa_sparse_attn_bwd_dense(const void* Q, const void* K, const void* V, const int32_t* idx,
                              const void* O, const float* lse, const void* dO, int B, int S,
                              int H, int Hkv, int Dqk, int Dv, int k, float scale, void* dQ,
                              void* dK, void* dV, void* ws, size_t ws_bytes, void* stream) {
  return attn_bwd_impl(Q, K, V, idx, O, lse, dO, B, S, H, Hkv, Dqk, Dv, k, scale, dQ, dK, dV, ws,
                       ws_bytes, stream, dsa::kBwdPathDense);
}

int dsa_sparse_attn_bwd_kernel(int B, int S, int H, int Hkv, int Dqk, int Dv, int k,
                               float scale) {
  if (B < 1 || S < 1 || H < 1 || k < 1) return -DSA_ERR_INVALID_ARG;
  if (Hkv < 1 || H % Hkv != 0) return -DSA_ERR_INVALID_ARG;
  if (H > 128 || !dsa::attn_dims_supported(Dqk, Dv)) return -DSA_ERR_UNSUPPORTED;
  return dsa::attn_bwd_kernel_kind(B, S, H, Dqk, Dv, k, scale, Hkv);
}


size_t dsa_index_topk_workspace_size(int B, int S, int block_rows) {
  if (B < 1 || S < 1 || block_rows < 1) return 0;
  const long long ld = (static_cast<long long>(S) + 3) / 4 * 4;
  const long long rows = block_rows < S ? block_rows : S;
  return static_cast<size_t>(B) * rows * ld * sizeof(float);
}

}  // extern "C"

namespace {

int index_topk_impl(const void* q_idx, const void* k_idx, const float* k_scale, const void* w,
                    int w_dtype, const int32_t* seg, int B, int S, int Hi, int Di, int k,
                    int block_rows, int32_t* idx, int32_t* count, float* vals, void* ws,
                    size_t ws_bytes, void* stream, int fp8) {
  if (!q_idx || !k_idx || !w || !idx) return DSA_ERR_INVALID_ARG;
  if (vals && !aligned16(vals)) return DSA_ERR_INVALID_ARG;
  if (k_scale && !aligned16(k_scale)) return DSA_ERR_INVALID_ARG;
  if (fp8 && Di % 16 != 0) return DSA_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || Hi < 1 || Di < 1 || k < 1) return DSA_ERR_INVALID_ARG;
  if (block_rows < 256 || block_rows % 256 != 0) return DSA_ERR_INVALID_ARG;
  if (w_dtype != DSA_F32 && w_dtype != DSA_BF16) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(w) || !aligned16(idx) ||
      (count && !aligned16(count)) || (seg && !aligned16(seg)))
    return DSA_ERR_INVALID_ARG;
  if (Di % 8 != 0) return DSA_ERR_INVALID_ARG;
  if (!dsa::indexer_dims_supported(Hi, Di)) return DSA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * S * Hi >= (1LL << 31)) return DSA_ERR_UNSUPPORTED;
  const size_t need = dsa_index_topk_workspace_size(B, S, block_rows);
  if (!ws || ws_bytes < need || !aligned16(ws)) return DSA_ERR_WORKSPACE;
  const long long ld = (static_cast<long long>(S) + 3) / 4 * 4;
  const int R = block_rows < S ? block_rows : S;
  float* buf = static_cast<float*>(ws);
  for (int t_lo = 0; t_lo < S; t_lo += R) {
    const int t_hi = t_lo + R < S ? t_lo + R : S;
    int rc = dsa::launch_index_scores_rows(q_idx, k_idx, w, w_dtype == DSA_BF16, seg, B, S, Hi,
                                           Di, buf, ld, as_stream(stream), fp8, k_scale, t_lo,
                                           t_hi, R);
    if (rc != DSA_OK) return rc;
    rc = dsa::launch_topk_rows(buf, ld, seg, B, S, k, idx, count, vals, as_stream(stream), t_lo,
                               t_hi, R);
    if (rc != DSA_OK) return rc;
  }
  return DSA_OK;
}

}  // namespace

extern "C" {

int dsa_index_topk(const void* q_idx, const void* k_idx, const void* w, int w_dtype,
                   const int32_t* seg, int B, int S, int Hi, int Di, int k, int block_rows,
                   int32_t* idx, int32_t* count, float* vals, void* ws, size_t ws_bytes,
                   void* stream) {
  return index_topk_impl(q_idx, k_idx, nullptr, w, w_dtype, seg, B, S, Hi, Di, k, block_rows,
                         idx, count, vals, ws, ws_bytes, stream, 0);
}

int dsa_index_topk_fp8(const void* q_idx, const void* k_idx, const float* k_scale, const void* w,
                       int w_dtype, const int32_t* seg, int B, int S, int Hi, int Di, int k,
                       int block_rows, int32_t* idx, int32_t* count, float* vals, void* ws,
                       size_t ws_bytes, void* stream) {
  return index_topk_impl(q_idx, k_idx, k_scale, w, w_dtype, seg, B, S, Hi, Di, k, block_rows,
                         idx, count, vals, ws, ws_bytes, stream, 1);
}

}  // extern "C"

namespace {

// the streaming form's workspace: sample scores, window thresholds, list counts, window
// lists, block flags and one block of rows of scores for the rows the lists do not settle
struct StreamLayout {
  size_t sample, thr, cnt, win, flags, buf, bytes;
};

size_t r256(size_t n) { return (n + 255) / 256 * 256; }

StreamLayout stream_layout(int B, int S, int block_rows) {
  StreamLayout ly = {0, 0, 0, 0, 0, 0, 0};
  if (B < 1 || S < 1 || block_rows < 1) return ly;
  const size_t rows = static_cast<size_t>(B) * S;
  const size_t ld = (static_cast<size_t>(S) + 3) / 4 * 4;
  const size_t R = block_rows < S ? block_rows : S;
  const size_t nblk = (static_cast<size_t>(S) + R - 1) / R;
  ly.sample = 0;
  ly.thr = r256(rows * dsa::kSampleKeys * sizeof(float));
  ly.cnt = ly.thr + r256(rows * 2 * sizeof(float));
  ly.win = ly.cnt + r256(rows * 4 * sizeof(int));
  ly.flags = ly.win + r256(rows * dsa::kStreamWindowCap * sizeof(int2));
  ly.buf = ly.flags + r256(nblk * sizeof(int));
  ly.bytes = ly.buf + r256(static_cast<size_t>(B) * R * ld * sizeof(float));
  return ly;
}

int index_topk_stream_impl(const void* q_idx, const void* k_idx, const float* k_scale,
                           const void* w, int w_dtype, const int32_t* seg, int B, int S, int Hi,
                           int Di, int k, int block_rows, int32_t* idx, int32_t* count,
                           float* vals, void* ws, size_t ws_bytes, void* stream, int fp8) {
  if (!q_idx || !k_idx || !w || !idx) return DSA_ERR_INVALID_ARG;
  if (vals && !aligned16(vals)) return DSA_ERR_INVALID_ARG;
  if (k_scale && !aligned16(k_scale)) return DSA_ERR_INVALID_ARG;
  if (fp8 && Di % 16 != 0) return DSA_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || Hi < 1 || Di < 1 || k < 1) return DSA_ERR_INVALID_ARG;
  if (block_rows < 256 || block_rows % 256 != 0) return DSA_ERR_INVALID_ARG;
  if (w_dtype != DSA_F32 && w_dtype != DSA_BF16) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(w) || !aligned16(idx) ||
      (count && !aligned16(count)) || (seg && !aligned16(seg)))
    return DSA_ERR_INVALID_ARG;
  if (Di % 8 != 0) return DSA_ERR_INVALID_ARG;
  if (!dsa::indexer_dims_supported(Hi, Di)) return DSA_ERR_UNSUPPORTED;
  if (S > dsa::kStreamMaxS || static_cast<long long>(B) * S * Hi >= (1LL << 31))
    return DSA_ERR_UNSUPPORTED;
  if (vals && k > 2048) return DSA_ERR_UNSUPPORTED;   // the finish stages scores by slot
  const StreamLayout ly = stream_layout(B, S, block_rows);
  if (!ws || ws_bytes < ly.bytes || !aligned16(ws)) return DSA_ERR_WORKSPACE;
  uint8_t* base = static_cast<uint8_t*>(ws);
  float* sample = reinterpret_cast<float*>(base + ly.sample);
  float* thr = reinterpret_cast<float*>(base + ly.thr);
  int* cnt = reinterpret_cast<int*>(base + ly.cnt);
  int2* win = reinterpret_cast<int2*>(base + ly.win);
  int* flags = reinterpret_cast<int*>(base + ly.flags);
  float* buf = reinterpret_cast<float*>(base + ly.buf);
  const cudaStream_t st = as_stream(stream);
  const long long rows = static_cast<long long>(B) * S;
  const int R = block_rows < S ? block_rows : S;
  const int nblk = (S + R - 1) / R;
  const int wb = w_dtype == DSA_BF16;
  if (cudaMemsetAsync(cnt, 0, static_cast<size_t>(rows) * 4 * sizeof(int), st) != cudaSuccess ||
      cudaMemsetAsync(flags, 0, static_cast<size_t>(nblk) * sizeof(int), st) != cudaSuccess)
    return DSA_ERR_CUDA;
  int rc = dsa::launch_index_sample(q_idx, k_idx, w, wb, seg, B, S, Hi, Di, st, fp8, k_scale,
                                    sample);
  if (rc == DSA_OK) rc = dsa::launch_stream_window(sample, seg, B, S, 256 / Hi, k, thr, st);
  if (rc == DSA_OK)
    rc = dsa::launch_index_emit(q_idx, k_idx, w, wb, seg, B, S, Hi, Di, st, fp8, k_scale, thr,
                                cnt, idx, vals, k, win, dsa::kStreamWindowCap);
  if (rc == DSA_OK)
    rc = dsa::launch_stream_finish(seg, B, S, k, cnt, win, dsa::kStreamWindowCap, idx, count,
                                   vals, flags, R, st);
  // the rows the lists did not settle: their blocks again through the memory form, each
  // launch gated on its block's flag on the device
  const long long ld = (static_cast<long long>(S) + 3) / 4 * 4;
  for (int bi = 0; rc == DSA_OK && bi < nblk; ++bi) {
    const int t_lo = bi * R, t_hi = t_lo + R < S ? t_lo + R : S;
    rc = dsa::launch_index_scores_rows(q_idx, k_idx, w, wb, seg, B, S, Hi, Di, buf, ld, st, fp8,
                                       k_scale, t_lo, t_hi, R, flags + bi);
    if (rc == DSA_OK)
      rc = dsa::launch_topk_rows(buf, ld, seg, B, S, k, idx, count, vals, st, t_lo, t_hi, R,
                                 flags + bi);
  }
  return rc;
}

}  // namespace

extern "C" {

size_t dsa_index_topk_stream_workspace_size(int B, int S, int block_rows) {
  return stream_layout(B, S, block_rows).bytes;
}

int dsa_index_topk_stream(const void* q_idx, const void* k_idx, const void* w, int w_dtype,
                          const int32_t* seg, int B, int S, int Hi, int Di, int k, int block_rows,
                          int32_t* idx, int32_t* count, float* vals, void* ws, size_t ws_bytes,
                          void* stream) {
  return index_topk_stream_impl(q_idx, k_idx, nullptr, w, w_dtype, seg, B, S, Hi, Di, k,
                                block_rows, idx, count, vals, ws, ws_bytes, stream, 0);
}

int dsa_index_topk_stream_fp8(const void* q_idx, const void* k_idx, const float* k_scale,
                              const void* w, int w_dtype, const int32_t* seg, int B, int S, int Hi,
                              int Di, int k, int block_rows, int32_t* idx, int32_t* count,
                              float* vals, void* ws, size_t ws_bytes, void* stream) {
  return index_topk_stream_impl(q_idx, k_idx, k_scale, w, w_dtype, seg, B, S, Hi, Di, k,
                                block_rows, idx, count, vals, ws, ws_bytes, stream, 1);
}

int dsa_indexer_loss(const void* Q, const void* K, const int32_t* idx, const float* lse,
                     const float* scores, int64_t ld_scores, int B, int S, int H, int Hkv,
                     int Dqk, int k, float scale, float grad_scale, float* kl, float* dI,
                     void* stream) {
  if (!Q || !K || !idx || !lse || !scores || !kl || !dI) return DSA_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || H < 1 || Hkv < 1 || Dqk < 1 || k < 1) return DSA_ERR_INVALID_ARG;
  // ld_scores = 0: scores holds the selected keys' scores slot by slot ([B, S, k])
  if (H % Hkv != 0 || ld_scores < 0 || (ld_scores > 0 && ld_scores < S))
    return DSA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(idx) || !aligned16(lse) ||
      !aligned16(scores) || !aligned16(kl) || !aligned16(dI))
    return DSA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * S >= (1LL << 31)) return DSA_ERR_UNSUPPORTED;
  if (Hkv == 1 && dsa::indexer_loss_supported(H, Dqk, scale))
    return dsa::launch_indexer_loss(Q, K, idx, lse, scores, ld_scores, B, S, H, Dqk, k, scale,
                                    grad_scale, kl, dI, as_stream(stream));
  return dsa::launch_indexer_loss_simt(Q, K, idx, lse, scores, ld_scores, B, S, H, Hkv, Dqk, k,
                                       scale, grad_scale, kl, dI, as_stream(stream));
}

int dsa_indexer_loss_bwd(const void* q_idx, const void* k_idx, const float* w,
                         const int32_t* idx, const float* dI, int B, int S, int Hi, int Di,
                         int k, float* dq_idx, float* dk_idx, float* dw, void* stream) {
  if (!q_idx || !k_idx || !w || !idx || !dI || !dq_idx || !dk_idx || !dw)
    return DSA_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || Hi < 1 || Di < 1 || k < 1) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(w) || !aligned16(idx) ||
      !aligned16(dI) || !aligned16(dq_idx) || !aligned16(dk_idx) || !aligned16(dw))
    return DSA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * S >= (1LL << 31)) return DSA_ERR_UNSUPPORTED;
  if (dsa::indexer_loss_bwd_supported(Hi, Di))
    return dsa::launch_indexer_loss_bwd(q_idx, k_idx, w, idx, dI, B, S, Hi, Di, k, dq_idx, dk_idx,
                                        dw, as_stream(stream));
  return dsa::launch_indexer_loss_bwd_simt(q_idx, k_idx, w, idx, dI, B, S, Hi, Di, k, dq_idx,
                                           dk_idx, dw, as_stream(stream));
}

}  // extern "C"
