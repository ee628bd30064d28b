// Lightning-indexer scores on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
//   I[b,t,s] = sum_h w[b,t,h] * max(0, q_idx[b,t,h,:] . k_idx[b,s,:])     (valid s <= t)
//
// ("DeepSeek3.2: Onboard sparse attention", Background: the indexer's per-head
// q.k product; "Implement QK attention head chunking for CSA", Description:
// per-head products reduced over heads. The per-head [S, S] products that the
// pages materialise and chunk never exist here: they live in TMEM for one tile
// and are reduced in registers.)
//
// Tiling. One UMMA tile is D[128 keys, 256 cols] = K_blk[128, Di] x Q_grp[256, Di]^T,
// where the 256 columns are G = 256/Hi consecutive queries x Hi heads (the rows of
// q_idx are already laid out that way). Each TMEM lane is one key, so the
// epilogue's sum over heads is a reduction inside one thread, and the scores of
// 32 consecutive keys of one query row leave as one coalesced 128-byte store.
//
// Persistent, warp-specialised CTA (one per SM):
//   warp 0     TMA producer: Q group tile (2 slots) and key tiles (3-stage ring)
//   warp 1     TMEM allocator and single-thread UMMA issuer (2 accumulators of 256 cols)
//   warps 2-9  epilogue: tcgen05.ld, ReLU, x w, sum over heads, mask, store
// Work item = (batch, query group); key blocks 0..t_max/128 of the item stream
// through the ring. Items are handed out heaviest first, strided over CTAs.
//
// FP8 form ("DeepSeek3.2: Onboard sparse attention", unit tests: the original
// indexer runs as an fp8 kernel on quantized activations): q_idx / k_idx as e4m3
// bytes on kind::f8f6f4 (K = 32 per instruction, twice the bf16 rate), and an
// optional positive scale per key. Since ReLU is positively homogeneous,
//   sum_h w * max(0, q . (c_s k)) = c_s * sum_h w * max(0, q . k),
// so the scale multiplies the reduced score; a per-(query, head) scale of q
// belongs in w.

#include <cuda.h>
#include <cuda_bf16.h>

#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kKeysPerTile = 128;  // UMMA M (TMEM lanes)
constexpr int kColsPerTile = 256;  // UMMA N
constexpr int kKStages = 3;
constexpr int kQSlots = 2;
constexpr int kAccBufs = 2;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + kEpiWarps * 32;
constexpr int kErr = DSA_STAGE_INDEXER | DSA_DEVERR_TIMEOUT;
constexpr int kModeStore = 0, kModeSample = 1, kModeEmit = 2;
// emit mode: items of at most this many queries (Hi >= 16) count their lists in shared
// memory and store the counts once per item; others add into global memory per warp
constexpr int kEmitSmemQueries = 16;

struct IndexerParams {
  int B, S, Di;
  int G;          // queries per tile (256 / Hi)
  int n_groups;   // ceil(S / G)
  int g_lo, g_hi; // the query groups of this launch (all of them, or one block of rows)
  int n_items;    // B * (g_hi - g_lo)
  int t_base;     // the first query row of the launch: row t is stored at row t - t_base
  int t_end;      // one past its last query row
  long long rows_blk;   // rows per batch of the score buffer
  int atom;       // K elements per swizzled row segment
  int n_atoms;    // Di / atom
  uint32_t atom_bytes;   // bytes of one swizzled row segment (32, 64 or 128)
  uint32_t layout;
  uint32_t q_slot_bytes, k_stage_bytes;
  const void* w;
  int w_bf16;
  const int32_t* seg;
  const float* k_scale;   // fp8 form: per-key scale [B, S] or nullptr
  float* scores;
  long long ld;
  int* err;
  int mode;               // kModeStore, kModeSample or kModeEmit
  const int* gate;        // non-null: the launch does nothing unless *gate != 0
  // kModeSample: the scores of up to kSampleTiles evenly spaced key tiles of each row
  float* sample;          // [B * S, kSampleKeys], NaN where the key is not valid
  // kModeEmit: per row, keys scoring >= U into `above` and keys in [L, U) into `win`
  const float* thr;       // [B * S, 2]: U, L (NaN: none)
  int* cnt;               // [B * S, 4]: keys >= U, keys in [L, U), valid keys (with seg)
  int32_t* above;         // [B * S, k]
  float* above_vals;      // null, or [B * S, k]: the scores beside the `above` entries
  int2* win;              // [B * S, cw]: (key index, score bits)
  int k, cw;
};

struct SmemTail {
  float w_s[kQSlots][kColsPerTile];  // head weights of the item, one slot per Q slot
  uint64_t q_full[kQSlots], q_empty[kQSlots];
  uint64_t w_full[kQSlots], w_empty[kQSlots];
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t acc_full[kAccBufs], acc_empty[kAccBufs];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int ecnt[kQSlots][kEmitSmemQueries][4];   // emit mode: list counters per item slot and query
};

__device__ __forceinline__ void item_coords(const IndexerParams& p, int item, int& b, int& t0,
                                            int& nkb) {
  // heaviest items (largest t) first
  const int gi = item / p.B;
  b = item - gi * p.B;
  const int g = p.g_hi - 1 - gi;
  t0 = g * p.G;
  int t_last = t0 + p.G - 1;
  if (t_last > p.S - 1) t_last = p.S - 1;
  nkb = t_last / kKeysPerTile + 1;
}

// Key tiles an item runs: all nkb of them, or (sample mode) sample_tiles(nkb) evenly spaced
// ones; tile_at(m) is the m-th (sample_tile), increasing in m.
template <int MODE>
__device__ __forceinline__ int item_tiles(int nkb) {
  return MODE == kModeSample ? sample_tiles(nkb) : nkb;
}
template <int MODE>
__device__ __forceinline__ int tile_at(int m, int nt, int nkb) {
  return MODE == kModeSample ? sample_tile(m, nt, nkb) : m;
}

// Emit mode, for one query row and the 32 keys of a warp (lane = key): keys scoring >= U
// join the row's `above` list, keys in [L, U) its window list, one atomic per list and
// warp; with segment ids the valid keys are counted too. Warp-collective.
__device__ __forceinline__ void emit_keys(const IndexerParams& p, long long row, int* cnt, int s,
                                          float val, bool valid, int lane) {
  const float2 ul = __ldg(reinterpret_cast<const float2*>(p.thr) + row);   // (U, L)
  const float U = ul.x, L = ul.y;
  const bool above = valid && val >= U;
  const bool win = valid && val >= L && !(val >= U);
  const uint32_t lt = (1u << lane) - 1u;
  uint32_t bal = __ballot_sync(0xffffffffu, above);
  if (bal) {
    int base = 0;
    if (lane == 0) base = atomicAdd(cnt, __popc(bal));
    base = __shfl_sync(0xffffffffu, base, 0);
    const int pos = base + __popc(bal & lt);
    if (above && pos < p.k) {
      p.above[row * p.k + pos] = s;
      if (p.above_vals) p.above_vals[row * p.k + pos] = val;
    }
  }
  bal = __ballot_sync(0xffffffffu, win);
  if (bal) {
    int base = 0;
    if (lane == 0) base = atomicAdd(cnt + 1, __popc(bal));
    base = __shfl_sync(0xffffffffu, base, 0);
    const int pos = base + __popc(bal & lt);
    if (win && pos < p.cw) p.win[row * p.cw + pos] = make_int2(s, __float_as_int(val));
  }
  if (p.seg != nullptr) {
    bal = __ballot_sync(0xffffffffu, valid);
    if (lane == 0 && bal) atomicAdd(cnt + 2, __popc(bal));
  }
}

// Emit mode for the NQ queries of one epilogue warp and the 32 keys of its lanes (key s
// of this lane), after a tile: every list of every query reserves its slots at once
// (lane q for the keys >= U of query q, lane 8 + q for its window keys, lane 16 + q
// for its valid keys when there are segment ids), then each lane writes its entries.
// cnt[q][*] are the item's shared-memory counters of item query q0 + q. Warp-collective.
template <int NQ>
__device__ __forceinline__ void emit_tile(const IndexerParams& p, const float (&val)[NQ],
                                          int (*cnt)[4], int q0, int b, int t0, int s,
                                          int seg_s, int lane) {
  static_assert(NQ <= 8, "one lane per query and list");
  const uint32_t lt = (1u << lane) - 1u;
  bool fa[NQ], fw[NQ];
  uint32_t ba[NQ], bw[NQ];
  uint32_t mine = 0u;
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const int t = t0 + q0 + q;
    const bool in_t = t < p.t_end;   // the same for every lane of the warp
    const long long row = static_cast<long long>(b) * p.S + t;
    bool valid = false;
    float U = INFINITY, L = INFINITY;
    if (in_t) {
      valid = s <= t && (p.seg == nullptr || seg_s == __ldg(p.seg + b * p.S + t));
      const float2 ul = __ldg(reinterpret_cast<const float2*>(p.thr) + row);   // (U, L)
      U = ul.x;
      L = ul.y;
    }
    fa[q] = valid && val[q] >= U;
    fw[q] = valid && val[q] >= L && !(val[q] >= U);
    ba[q] = __ballot_sync(0xffffffffu, fa[q]);
    bw[q] = __ballot_sync(0xffffffffu, fw[q]);
    const uint32_t bv = p.seg != nullptr ? __ballot_sync(0xffffffffu, valid) : 0u;
    if (lane == q) mine = ba[q];
    if (lane == 8 + q) mine = bw[q];
    if (lane == 16 + q) mine = bv;
  }
  int base = 0;
  if (mine != 0u) base = atomicAdd(&cnt[q0 + (lane & 7)][lane >> 3], __popc(mine));
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const long long row = static_cast<long long>(b) * p.S + t0 + q0 + q;
    const int pa = __shfl_sync(0xffffffffu, base, q) + __popc(ba[q] & lt);
    const int pw = __shfl_sync(0xffffffffu, base, 8 + q) + __popc(bw[q] & lt);
    if (fa[q] && pa < p.k) {
      p.above[row * p.k + pa] = s;
      if (p.above_vals) p.above_vals[row * p.k + pa] = val[q];
    }
    if (fw[q] && pw < p.cw) p.win[row * p.cw + pw] = make_int2(s, __float_as_int(val[q]));
  }
}

// Drain wait used only at exit: ignores the abort flag, still bounded.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* err) {
  const uint32_t a = smem_u32(bar);
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      report_error(err, kErr);
      return;
    }
  }
}

__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// acc += a * b on both halves with one paired fp32 FMA (each half rounds as fmaf)
__device__ __forceinline__ void ffma2(float2& acc, float2 a, float2 b) {
  unsigned long long d, x, y;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b.x), "f"(b.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(acc.x), "f"(acc.y));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(x), "l"(y));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(acc.x), "=f"(acc.y) : "l"(d));
}

template <int HI, bool F8, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k, const IndexerParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  if (p.gate != nullptr && *reinterpret_cast<const volatile int*>(p.gate) == 0) return;
  // The swizzled tiles need 1024-byte alignment. The dynamic window starts
  // 1024-aligned when the kernel has no static shared memory; refuse to run
  // (and say so) rather than feed misaligned tiles to TMA / UMMA.
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) report_error(p.err, DSA_STAGE_INDEXER | DSA_DEVERR_MISALIGNED);
    return;
  }
  uint8_t* q_smem = smem;
  uint8_t* k_smem = q_smem + kQSlots * p.q_slot_bytes;
  SmemTail* tail = reinterpret_cast<SmemTail*>(k_smem + kKStages * p.k_stage_bytes);
  volatile int* abort_flag = &tail->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kQSlots; ++i) {
      mbar_init(&tail->q_full[i], 1);
      mbar_init(&tail->q_empty[i], 1);
      mbar_init(&tail->w_full[i], 32);
      mbar_init(&tail->w_empty[i], kEpiWarps);
    }
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&tail->k_full[i], 1);
      mbar_init(&tail->k_empty[i], 1);
    }
    for (int i = 0; i < kAccBufs; ++i) {
      mbar_init(&tail->acc_full[i], 1);
      mbar_init(&tail->acc_empty[i], kEpiWarps);
    }
    mbar_init(&tail->drain, 1);
    tail->abort_flag = 0;
    for (int i = 0; i < kQSlots * kEmitSmemQueries * 4; ++i) (&tail->ecnt[0][0][0])[i] = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
  }
  if (warp == 1) {
    tmem_alloc(&tail->tmem_base, kAccBufs * kColsPerTile);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tail->tmem_base;

  const uint32_t atom_bytes = p.atom_bytes;
  const uint32_t sbo = 8u * atom_bytes;
  // emit mode with few queries per item: the list counters live in shared memory, per item
  // slot; the producer stores an item's counts and zeroes them once every epilogue warp has
  // released the slot (w_empty), before the slot's next item
  constexpr bool kSmemCnt = MODE == kModeEmit && kColsPerTile / HI <= kEmitSmemQueries;
  constexpr int kEmitNqw = kSmemCnt ? 128 / HI : 1;   // queries of one epilogue warp's columns

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // All 32 lanes stage the head weights of each item; lane 0 issues the TMA copies.
    int ks = 0, qs = 0;
    uint32_t k_par = 1, q_par = 1;
    uint32_t k_issued[kKStages] = {0, 0, 0}, q_issued[kQSlots] = {0, 0};
    uint32_t k_last_par[kKStages] = {0, 0, 0}, q_last_par[kQSlots] = {0, 0};
    int slot_b[kQSlots] = {-1, -1}, slot_t0[kQSlots] = {0, 0};   // the item of each slot
    auto flush_counts = [&](int sl) {
      if constexpr (kSmemCnt) {
        if (slot_b[sl] < 0) return;
        for (int i = lane; i < (kColsPerTile / HI) * 3; i += 32) {
          const int q = i / 3, c = i - 3 * q, t = slot_t0[sl] + q;
          if (t < p.t_end)
            p.cnt[4 * (static_cast<long long>(slot_b[sl]) * p.S + t) + c] = tail->ecnt[sl][q][c];
          tail->ecnt[sl][q][c] = 0;
        }
        slot_b[sl] = -1;
      }
    };
    bool ok = true;
    for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x) {
      int b, t0, nkb;
      item_coords(p, item, b, t0, nkb);
      int okw = 1;
      if (lane == 0) okw = mbar_wait(&tail->w_empty[qs], q_par, abort_flag, p.err, kErr) ? 1 : 0;
      if (__shfl_sync(0xffffffffu, okw, 0) == 0) break;
      flush_counts(qs);   // the slot's previous item is finished
      slot_b[qs] = b;
      slot_t0[qs] = t0;
      for (int c = lane; c < kColsPerTile; c += 32) {
        const int tq = t0 + c / HI;
        float wv = 0.f;
        if (tq < p.S) {
          const long long off = (static_cast<long long>(b) * p.S + tq) * HI + (c % HI);
          wv = p.w_bf16 ? bf16_bits_to_float(static_cast<const uint16_t*>(p.w)[off])
                        : static_cast<const float*>(p.w)[off];
        }
        tail->w_s[qs][c] = wv;
      }
      mbar_arrive(&tail->w_full[qs]);
      if (lane == 0) {
        if (!mbar_wait(&tail->q_empty[qs], q_par, abort_flag, p.err, kErr)) ok = false;
        if (ok) {
          mbar_arrive_expect_tx(&tail->q_full[qs], p.q_slot_bytes);
          const int qrow = (b * p.S + t0) * HI;
          for (int a = 0; a < p.n_atoms; ++a)
            tma_load_2d(q_smem + qs * p.q_slot_bytes + a * kColsPerTile * atom_bytes, &tm_q,
                        &tail->q_full[qs], a * p.atom, qrow);
          q_issued[qs] = 1;
          q_last_par[qs] = q_par ^ 1u;
        }
        const int nt = item_tiles<MODE>(nkb);
        for (int m = 0; ok && m < nt; ++m) {
          const int j = tile_at<MODE>(m, nt, nkb);
          if (!mbar_wait(&tail->k_empty[ks], k_par, abort_flag, p.err, kErr)) { ok = false; break; }
          mbar_arrive_expect_tx(&tail->k_full[ks], p.k_stage_bytes);
          const int krow = b * p.S + j * kKeysPerTile;
          for (int a = 0; a < p.n_atoms; ++a)
            tma_load_2d(k_smem + ks * p.k_stage_bytes + a * kKeysPerTile * atom_bytes, &tm_k,
                        &tail->k_full[ks], a * p.atom, krow);
          k_issued[ks] = 1;
          k_last_par[ks] = k_par ^ 1u;
          if (++ks == kKStages) { ks = 0; k_par ^= 1u; }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (++qs == kQSlots) { qs = 0; q_par ^= 1u; }
    }
    // the counts of the items still in flight, once their slots are released
    for (int i = 0; kSmemCnt && ok && i < kQSlots; ++i) {
      if (slot_b[qs] >= 0) {
        int okw = 1;
        if (lane == 0) okw = mbar_wait(&tail->w_empty[qs], q_par, abort_flag, p.err, kErr) ? 1 : 0;
        if (__shfl_sync(0xffffffffu, okw, 0) == 0) break;
        flush_counts(qs);
      }
      if (++qs == kQSlots) { qs = 0; q_par ^= 1u; }
    }
    // Let every copy this warp started land before the CTA exits.
    if (lane == 0) {
      for (int i = 0; i < kQSlots; ++i)
        if (q_issued[i]) drain_wait(&tail->q_full[i], q_last_par[i], p.err);
      for (int i = 0; i < kKStages; ++i)
        if (k_issued[i]) drain_wait(&tail->k_full[i], k_last_par[i], p.err);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ UMMA issuer
    if (lane == 0) {
      const uint32_t idesc = F8 ? umma_idesc_e4m3(kKeysPerTile, kColsPerTile)
                                : umma_idesc_bf16(kKeysPerTile, kColsPerTile);
      const int ksteps_per_atom = static_cast<int>(atom_bytes / 32u);   // 32 bytes of K each
      int ks = 0, qs = 0, as = 0;
      uint32_t k_par = 0, q_par = 0, a_par = 1;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x) {
        int b, t0, nkb;
        item_coords(p, item, b, t0, nkb);
        if (!mbar_wait(&tail->q_full[qs], q_par, abort_flag, p.err, kErr)) { ok = false; break; }
        // base descriptors of the item's Q slot and (below) of each key stage, advanced by
        // constants per MMA: issue blocks at the pipe's pace, so scalar work per MMA would
        // leave the tensor pipe idle between instructions
        const uint64_t bdesc0 = umma_sdesc(smem_u32(q_smem + qs * p.q_slot_bytes), sbo, p.layout);
        const int nt = item_tiles<MODE>(nkb);
        for (int m = 0; m < nt; ++m) {
          if (!mbar_wait(&tail->k_full[ks], k_par, abort_flag, p.err, kErr)) { ok = false; break; }
          if (!mbar_wait(&tail->acc_empty[as], a_par, abort_flag, p.err, kErr)) { ok = false; break; }
          tc_fence_after();
          const uint64_t adesc0 = umma_sdesc(smem_u32(k_smem + ks * p.k_stage_bytes), sbo, p.layout);
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(as * kColsPerTile);
          auto mma = [&](uint64_t ad, uint64_t bd, uint32_t acc) {
            if (F8)
              umma_f8(d_tmem, ad, bd, idesc, acc);
            else
              umma_bf16(d_tmem, ad, bd, idesc, acc);
          };
          for (int a = 0; a < p.n_atoms; ++a) {
            const uint64_t ad = umma_desc_adv(adesc0, a * kKeysPerTile * atom_bytes);
            const uint64_t bd = umma_desc_adv(bdesc0, a * kColsPerTile * atom_bytes);
            if (ksteps_per_atom == 4) {   // 128-byte rows: four MMAs of 32 bytes of K each
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma(umma_desc_adv(ad, kk * 32u), umma_desc_adv(bd, kk * 32u), (a | kk) != 0 ? 1u : 0u);
            } else {
              for (int kk = 0; kk < ksteps_per_atom; ++kk)
                mma(umma_desc_adv(ad, kk * 32u), umma_desc_adv(bd, kk * 32u), (a | kk) != 0 ? 1u : 0u);
            }
          }
          umma_commit(&tail->k_empty[ks]);
          umma_commit(&tail->acc_full[as]);
          if (++ks == kKStages) { ks = 0; k_par ^= 1u; }
          if (++as == kAccBufs) { as = 0; a_par ^= 1u; }
        }
        if (!ok) break;
        umma_commit(&tail->q_empty[qs]);
        if (++qs == kQSlots) { qs = 0; q_par ^= 1u; }
      }
      // Every UMMA issued above has completed once this arrives.
      umma_commit(&tail->drain);
      drain_wait(&tail->drain, 0, p.err);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = warp - 2;              // 0..7
    const int quarter = warp & 3;        // TMEM lane quarter this warp may access
    const int half = e >> 2;             // which 128 of the 256 columns
    // The e4m3 kernel's MMAs take half the bf16 time, so its epilogue sets its pace: at 64
    // index heads its warps keep their 128 head weights in registers for a whole item (no
    // shared-memory weight loads per tile) and read TMEM 16 columns at a time to make room
    // for them. The bf16 kernel (waiting less on its epilogue) keeps the weights in shared
    // memory, and so do fewer heads, whose many queries per chunk leave no registers.
    constexpr bool kRegW = F8 && MODE == kModeStore && HI == 64;
    constexpr int CW = kRegW ? 16 : 32;           // columns per chunk (one TMEM load)
    constexpr int QPC = HI >= CW ? 1 : CW / HI;   // queries per chunk
    constexpr int CPQ = HI >= CW ? HI / CW : 1;   // chunks per query
    int as = 0, ws = 0;
    uint32_t a_par = 0, w_par = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x) {
      int b, t0, nkb;
      item_coords(p, item, b, t0, nkb);
      // head weights of this query group: column c = (query c / HI, head c % HI)
      if (!__all_sync(0xffffffffu, mbar_wait(&tail->w_full[ws], w_par, abort_flag, p.err, kErr))) break;
      const float* w_item = tail->w_s[ws];
      float wreg[kRegW ? 128 : 1];
      if constexpr (kRegW) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float4 w4 = *reinterpret_cast<const float4*>(w_item + half * 128 + 4 * i);
          wreg[4 * i] = w4.x;
          wreg[4 * i + 1] = w4.y;
          wreg[4 * i + 2] = w4.z;
          wreg[4 * i + 3] = w4.w;
        }
      }

      const int nt = item_tiles<MODE>(nkb);
      for (int m = 0; m < nt; ++m) {
        const int j = tile_at<MODE>(m, nt, nkb);
        if (!__all_sync(0xffffffffu, mbar_wait(&tail->acc_full[as], a_par, abort_flag, p.err, kErr))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int s = j * kKeysPerTile + quarter * 32 + lane;
        const int seg_s = (p.seg != nullptr && s < p.S) ? __ldg(p.seg + b * p.S + s) : 0;
        const float ks = (F8 && p.k_scale != nullptr && s < p.S) ? __ldg(p.k_scale + b * p.S + s) : 1.f;
        const uint32_t t_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                static_cast<uint32_t>(as * kColsPerTile + half * 128);
        // this warp's 128 columns as two pairs of 32-column chunks, two TMEM loads
        // per wait; heads h, h+1 of a query go through one paired fp32 FMA (even and
        // odd heads summed apart, then added)
        float2 acc2[QPC];
#pragma unroll
        for (int i = 0; i < QPC; ++i) acc2[i] = make_float2(0.f, 0.f);
        // emit mode with shared-memory counters: this warp's scores of the tile, one per
        // query, listed together after the tile (one atomic instruction for every list)
        float ev[kEmitNqw];
        auto chunk = [&](int ch, const uint32_t (&v)[CW]) {
          const float* wrow = w_item + half * 128 + ch * CW;
#pragma unroll
          for (int j4 = 0; j4 < CW; j4 += 4) {
            float4 w4;
            if constexpr (kRegW) {
              w4 = make_float4(wreg[ch * CW + j4], wreg[ch * CW + j4 + 1], wreg[ch * CW + j4 + 2],
                               wreg[ch * CW + j4 + 3]);
            } else {
              w4 = *reinterpret_cast<const float4*>(wrow + j4);   // 4 weights per load
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int jj = j4 + 2 * u;
              const float2 w2 = u == 0 ? make_float2(w4.x, w4.y) : make_float2(w4.z, w4.w);
              const float2 r2 = make_float2(fmaxf(__uint_as_float(v[jj]), 0.f),
                                            fmaxf(__uint_as_float(v[jj + 1]), 0.f));
              if (HI >= 2) {
                ffma2(acc2[jj / (CW / QPC)], r2, w2);
              } else {   // one head per query: every column is its own query
                acc2[jj].x = fmaf(w2.x, r2.x, acc2[jj].x);
                acc2[jj + 1].x = fmaf(w2.y, r2.y, acc2[jj + 1].x);
              }
            }
          }
          if ((ch + 1) % CPQ == 0) {
            const int cq = ch + 1 - CPQ;
#pragma unroll
            for (int i = 0; i < QPC; ++i) {
              const int qi = (half * 128 + cq * CW) / HI + i;
              const int t = t0 + qi;
              if (MODE == kModeStore) {
                if (t < p.t_end && s <= t) {
                  float val = acc2[i].x + acc2[i].y;
                  if (F8 && p.k_scale != nullptr) val *= ks;
                  if (p.seg != nullptr && seg_s != __ldg(p.seg + b * p.S + t)) val = -INFINITY;
                  p.scores[(static_cast<long long>(b) * p.rows_blk + (t - p.t_base)) * p.ld + s] =
                      val;
                }
                acc2[i] = make_float2(0.f, 0.f);
                continue;
              }
              const bool in_t = t < p.t_end;   // the same for every lane of the warp
              float val = acc2[i].x + acc2[i].y;
              if (F8 && p.k_scale != nullptr) val *= ks;
              const bool same_doc = p.seg == nullptr || !in_t || s > t ||
                                    seg_s == __ldg(p.seg + b * p.S + t);
              if (MODE == kModeSample) {
                if (in_t)
                  p.sample[(static_cast<long long>(b) * p.S + t) * kSampleKeys + m * kKeysPerTile +
                           quarter * 32 + lane] =
                      s <= t && same_doc ? val : __int_as_float(0x7fc00000);
              } else if constexpr (kSmemCnt) {
                (void)same_doc;
                ev[(cq * CW) / HI + i] = val;
              } else if (in_t) {
                const long long row = static_cast<long long>(b) * p.S + t;
                emit_keys(p, row, p.cnt + 4 * row, s, val, s <= t && same_doc, lane);
              }
              acc2[i] = make_float2(0.f, 0.f);
            }
          }
        };
        if constexpr (kRegW) {
#pragma unroll
          for (int ch = 0; ch < 128 / CW; ++ch) {
            uint32_t v[CW];
            tmem_ld_x16(t_base + ch * CW, v);
            tmem_ld_wait();
            chunk(ch, v);
          }
        } else {
#pragma unroll
          for (int pr = 0; pr < 2; ++pr) {
            uint32_t va[CW], vb[CW];
            tmem_ld_x32(t_base + (2 * pr) * 32, va);
            tmem_ld_x32(t_base + (2 * pr + 1) * 32, vb);
            tmem_ld_wait();
            chunk(2 * pr, va);
            chunk(2 * pr + 1, vb);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tail->acc_empty[as]);
        if (++as == kAccBufs) { as = 0; a_par ^= 1u; }
        if constexpr (kSmemCnt) emit_tile<kEmitNqw>(p, ev, tail->ecnt[ws], (half * 128) / HI, b,
                                                    t0, s, seg_s, lane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->w_empty[ws]);
      if (++ws == kQSlots) { ws = 0; w_par ^= 1u; }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kAccBufs * kColsPerTile);
}

// ----------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

bool make_map(CUtensorMap* map, const void* base, uint64_t rows, int cols, int box_cols,
              int box_rows, CUtensorMapSwizzle swz, bool f8) {
  EncodeTiledFn fn = get_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * (f8 ? 1 : 2)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int HI, bool F8, int MODE>
int launch_hi(const CUtensorMap& mq, const CUtensorMap& mk, const IndexerParams& p,
              size_t smem_bytes, cudaStream_t stream) {
  auto kern = indexer_kernel<HI, F8, MODE>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_bytes)) != cudaSuccess)
    return DSA_ERR_CUDA;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int grid = p.n_items < sms ? p.n_items : sms;
  if (grid < 1) grid = 1;
  kern<<<grid, kThreads, smem_bytes, stream>>>(mq, mk, p);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace

bool indexer_dims_supported(int Hi, int Di) {
  const bool hi_ok = Hi >= 1 && Hi <= 128 && (Hi & (Hi - 1)) == 0;
  const bool di_ok = Di == 32 || Di == 64 || Di == 128;
  return hi_ok && di_ok;
}

template <bool F8, int MODE>
int launch_hi_any(int Hi, const CUtensorMap& mq, const CUtensorMap& mk, const IndexerParams& p,
                  size_t smem_bytes, cudaStream_t stream) {
  switch (Hi) {
    case 1: return launch_hi<1, F8, MODE>(mq, mk, p, smem_bytes, stream);
    case 2: return launch_hi<2, F8, MODE>(mq, mk, p, smem_bytes, stream);
    case 4: return launch_hi<4, F8, MODE>(mq, mk, p, smem_bytes, stream);
    case 8: return launch_hi<8, F8, MODE>(mq, mk, p, smem_bytes, stream);
    case 16: return launch_hi<16, F8, MODE>(mq, mk, p, smem_bytes, stream);
    case 32: return launch_hi<32, F8, MODE>(mq, mk, p, smem_bytes, stream);
    case 64: return launch_hi<64, F8, MODE>(mq, mk, p, smem_bytes, stream);
    case 128: return launch_hi<128, F8, MODE>(mq, mk, p, smem_bytes, stream);
    default: return DSA_ERR_UNSUPPORTED;
  }
}

template <bool F8>
int launch_mode(int Hi, const CUtensorMap& mq, const CUtensorMap& mk, const IndexerParams& p,
                size_t smem_bytes, cudaStream_t stream) {
  if (p.mode == kModeSample)
    return launch_hi_any<F8, kModeSample>(Hi, mq, mk, p, smem_bytes, stream);
  if (p.mode == kModeEmit) return launch_hi_any<F8, kModeEmit>(Hi, mq, mk, p, smem_bytes, stream);
  return launch_hi_any<F8, kModeStore>(Hi, mq, mk, p, smem_bytes, stream);
}

int launch_index_scores(const void* q_idx, const void* k_idx, const void* w, int w_is_bf16,
                        const int32_t* seg, int B, int S, int Hi, int Di, float* scores,
                        int64_t ld, cudaStream_t stream, int fp8, const float* k_scale) {
  return launch_index_scores_rows(q_idx, k_idx, w, w_is_bf16, seg, B, S, Hi, Di, scores, ld,
                                  stream, fp8, k_scale, 0, S, S);
}

namespace {

// the launch of one indexer pass; `extra` carries the mode and its buffers
int launch_pass(const void* q_idx, const void* k_idx, const void* w, int w_is_bf16,
                const int32_t* seg, int B, int S, int Hi, int Di, float* scores, int64_t ld,
                cudaStream_t stream, int fp8, const float* k_scale, int t_lo, int t_hi,
                long long rows_blk, const IndexerParams& extra) {
  IndexerParams p = extra;
  p.B = B;
  p.S = S;
  p.Di = Di;
  p.G = kColsPerTile / Hi;
  p.n_groups = (S + p.G - 1) / p.G;
  // t_lo is a multiple of G (the callers' blocks are multiples of 256 rows)
  p.g_lo = t_lo / p.G;
  p.g_hi = (t_hi + p.G - 1) / p.G;
  p.n_items = B * (p.g_hi - p.g_lo);
  p.t_base = t_lo;
  p.t_end = t_hi < S ? t_hi : S;
  p.rows_blk = rows_blk;
  // one swizzled row segment holds up to 128 bytes of K: 64 bf16 or 128 e4m3 values
  const int ebytes = fp8 ? 1 : 2;
  p.atom = Di * ebytes >= 128 ? 128 / ebytes : Di;
  p.n_atoms = Di / p.atom;
  p.atom_bytes = static_cast<uint32_t>(p.atom * ebytes);
  CUtensorMapSwizzle swz;
  if (p.atom_bytes == 128) {
    p.layout = kLayoutSw128;
    swz = CU_TENSOR_MAP_SWIZZLE_128B;
  } else if (p.atom_bytes == 64) {
    p.layout = kLayoutSw64;
    swz = CU_TENSOR_MAP_SWIZZLE_64B;
  } else {
    p.layout = kLayoutSw32;
    swz = CU_TENSOR_MAP_SWIZZLE_32B;
  }
  p.q_slot_bytes = static_cast<uint32_t>(kColsPerTile) * Di * ebytes;
  p.k_stage_bytes = static_cast<uint32_t>(kKeysPerTile) * Di * ebytes;
  p.w = w;
  p.w_bf16 = w_is_bf16;
  p.seg = seg;
  p.k_scale = k_scale;
  p.scores = scores;
  p.ld = ld;
  p.err = device_error_word();

  CUtensorMap mq, mk;
  if (!make_map(&mq, q_idx, static_cast<uint64_t>(B) * S * Hi, Di, p.atom, kColsPerTile, swz,
                fp8 != 0))
    return DSA_ERR_CUDA;
  if (!make_map(&mk, k_idx, static_cast<uint64_t>(B) * S, Di, p.atom, kKeysPerTile, swz,
                fp8 != 0))
    return DSA_ERR_CUDA;

  const size_t smem_bytes = kQSlots * static_cast<size_t>(p.q_slot_bytes) +
                            kKStages * static_cast<size_t>(p.k_stage_bytes) + sizeof(SmemTail);
  return fp8 ? launch_mode<true>(Hi, mq, mk, p, smem_bytes, stream)
             : launch_mode<false>(Hi, mq, mk, p, smem_bytes, stream);
}

IndexerParams no_extra() {
  IndexerParams e = {};
  e.mode = kModeStore;
  return e;
}

}  // namespace

int launch_index_scores_rows(const void* q_idx, const void* k_idx, const void* w, int w_is_bf16,
                             const int32_t* seg, int B, int S, int Hi, int Di, float* scores,
                             int64_t ld, cudaStream_t stream, int fp8, const float* k_scale,
                             int t_lo, int t_hi, long long rows_blk, const int* gate) {
  IndexerParams e = no_extra();
  e.gate = gate;
  return launch_pass(q_idx, k_idx, w, w_is_bf16, seg, B, S, Hi, Di, scores, ld, stream, fp8,
                     k_scale, t_lo, t_hi, rows_blk, e);
}

int launch_index_sample(const void* q_idx, const void* k_idx, const void* w, int w_is_bf16,
                        const int32_t* seg, int B, int S, int Hi, int Di, cudaStream_t stream,
                        int fp8, const float* k_scale, float* sample) {
  IndexerParams e = no_extra();
  e.mode = kModeSample;
  e.sample = sample;
  return launch_pass(q_idx, k_idx, w, w_is_bf16, seg, B, S, Hi, Di, nullptr, 0, stream, fp8,
                     k_scale, 0, S, S, e);
}

int launch_index_emit(const void* q_idx, const void* k_idx, const void* w, int w_is_bf16,
                      const int32_t* seg, int B, int S, int Hi, int Di, cudaStream_t stream,
                      int fp8, const float* k_scale, const float* thr, int* cnt, int32_t* above,
                      float* above_vals, int k, int2* win, int cw) {
  IndexerParams e = no_extra();
  e.mode = kModeEmit;
  e.thr = thr;
  e.cnt = cnt;
  e.above = above;
  e.above_vals = above_vals;
  e.k = k;
  e.win = win;
  e.cw = cw;
  return launch_pass(q_idx, k_idx, w, w_is_bf16, seg, B, S, Hi, Di, nullptr, 0, stream, fp8,
                     k_scale, 0, S, S, e);
}

}  // namespace dsa
