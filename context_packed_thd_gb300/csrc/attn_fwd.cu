// Causal packed-THD attention forward on tcgen05 tensor cores (sm_103a).
//
// What is computed (TransformerEngine PR #3221, "Scope and constraints" and
// "What changed"): causal THD self-attention without a sliding window, one
// context-parallel rank's query slice against the full (all-gathered) K/V
// buffer, documents isolated through cu_seqlens / cu_seqlens_padded. Output
// O in bf16 and the natural-log LSE in fp32 ([Hq, t_local]).
//
// Kernel design (one CTA per (128-row query tile, query head)):
//  * warp 0  -- TMA producer: Q tile once, then K and V 128-key blocks into a
//               two-stage shared-memory ring (128-byte swizzle, the layout the
//               UMMA descriptors read).
//  * warp 1  -- owns the 512-column TMEM allocation; one lane issues the
//               tcgen05 MMAs: S_i = Q K_i^T into one of two TMEM S buffers,
//               then O += P_{i-1} V_{i-1} into the TMEM O accumulator.
//  * warps 2..5 -- softmax: each thread owns one query row (its TMEM lane),
//               reads S_i with tcgen05.ld, masks by the row's key interval
//               [doc start, own position] clipped to the end of the tile
//               interval the block belongs to (only on blocks that the
//               tile's bounds do not cover fully), keeps the fp32 running max / sum
//               in base 2, rescales O in TMEM only when the max grows by more
//               than 2^8 (the result is exact either way), writes P as bf16
//               into swizzled shared memory and hands it to the MMA lane.
//               At the end it normalises O and writes out and LSE.
// Key blocks start at the tile's interval starts (document starts), so
// whole documents that a tile does not see are never loaded or multiplied.
// The grid runs the tiles in decreasing-cost order.
#include <cuda_bf16.h>

#include "attn_meta.cuh"
#include "common.cuh"
#include "sm100.cuh"

namespace cpthd {

using namespace sm100;

constexpr int kAttnThreads = 192;
constexpr int kStages = 2;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 256x

template <int D>
struct AttnSmem {
  static constexpr int kChunk = kBlockM * 64 * 2;      // one 128-row x 64-column bf16 swizzle panel
  static constexpr int kChunks = D / 64;
  static constexpr int kQ = kChunks * kChunk;          // Q tile
  static constexpr int kKV = kChunks * kChunk;         // one K or V block
  static constexpr int kP = 2 * kChunk;                // P: 128 rows x 128 keys
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQ;
  static constexpr int kVOff = kKOff + kStages * kKV;
  static constexpr int kPOff = kVOff + kStages * kKV;
  static constexpr int kBytes = kPOff + kP;
  // request at least this much so that one CTA holds an SM (TMEM is taken whole)
  static constexpr int kLaunchBytes = (kBytes + 1024 > 120 * 1024) ? kBytes + 1024 : 120 * 1024;
};

struct AttnParams {
  const int32_t* row_lo;
  const int32_t* row_hi;
  const TileInfo* tile_info;
  const int2* intervals;
  const int32_t* order;
  __nv_bfloat16* out;
  float* lse;
  long long t_local;
  int Hq;
  int Hkv;
  int max_blocks;  // upper bound on blocks per tile, guards malformed metadata
  float scale_log2;
  int32_t* err;
};

// Walks the key blocks of a tile: interval by interval, 128 keys at a time.
struct BlockCursor {
  const int2* iv;
  int n_iv;
  int k;      // interval index
  int start;  // start key of the current block
  int end;    // end key (inclusive) of the current interval
  __device__ void init(const int2* intervals, int n) {
    iv = intervals;
    n_iv = n;
    k = 0;
    if (n > 0) { int2 a = iv[0]; start = a.x; end = a.y; } else { start = 0; end = -1; }
  }
  __device__ void next() {
    start += kBlockN;
    if (start > end && ++k < n_iv) { int2 a = iv[k]; start = a.x; end = a.y; }
  }
};

__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  int local_abort = 0;
  return mbar_wait(bar, parity, &local_abort);
}

// All lanes of a warp wait; the outcome is made warp-uniform so that the
// .sync.aligned TMEM instructions that follow run on the whole warp or not at all.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using L = AttnSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + L::kQOff;
  uint8_t* sK = smem + L::kKOff;
  uint8_t* sV = smem + L::kVOff;
  uint8_t* sP = smem + L::kPOff;

  __shared__ uint64_t q_full, k_full[kStages], v_full[kStages], k_empty[kStages], v_empty[kStages];
  __shared__ uint64_t s_full[2], s_free[2], p_full, o_done, drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.x;
  const int tile = __ldg(p.order + item / p.Hq);
  const int h = item % p.Hq;
  const int kvh = h / (p.Hq / p.Hkv);
  const TileInfo ti = p.tile_info[tile];
  const int n_blocks = min(max(ti.n_blocks, 0), p.max_blocks);
  const int2* tile_iv = p.intervals + static_cast<long long>(tile) * kBlockM;
  const int n_iv = min(max(ti.n_intervals, 0), kBlockM);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], 4);
    }
    mbar_init(&p_full, 4);
    mbar_init(&o_done, 1);
    mbar_init(&drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t tmem_s0 = tmem;         // S buffers: columns [0,128) and [128,256)
  const uint32_t tmem_o = tmem + 256;    // O accumulator: columns [256, 256 + D)

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_blocks > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&q_full, L::kQ);
      for (int c = 0; c < L::kChunks; ++c) tma_load_3d(sQ + c * L::kChunk, &tm_q, &q_full, c * 64, h, tile * kBlockM);
      BlockCursor cur;
      cur.init(tile_iv, n_iv);
      int issued = 0;
      for (int i = 0; i < n_blocks; ++i) {
        const int st = i & 1;
        const uint32_t par = ((i >> 1) + 1) & 1;
        if (i >= kStages && !mbar_wait(&k_empty[st], par, &abort_flag)) break;
        mbar_arrive_expect_tx(&k_full[st], L::kKV);
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(sK + st * L::kKV + c * L::kChunk, &tm_k, &k_full[st], c * 64, kvh, cur.start);
        if (i >= kStages && !mbar_wait(&v_empty[st], par, &abort_flag)) { issued = 2 * i + 1; break; }
        mbar_arrive_expect_tx(&v_full[st], L::kKV);
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(sV + st * L::kKV + c * L::kChunk, &tm_v, &v_full[st], c * 64, kvh, cur.start);
        issued = 2 * i + 2;
        cur.next();
      }
      if (abort_flag) {
        // let every copy still in flight land before the CTA exits
        mbar_wait_drain(&q_full, 0);
        for (int x = (issued > 4 ? issued - 4 : 0); x < issued; ++x) {
          const int i = x >> 1, st = i & 1;
          mbar_wait_drain((x & 1) ? &v_full[st] : &k_full[st], (i >> 1) & 1);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_blocks > 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kBlockM, kBlockN, 0, 0);
      constexpr uint32_t kIdescO = idesc_bf16_f32(kBlockM, D, 0, 1);
      const uint32_t q0 = smem_u32(sQ), k0 = smem_u32(sK), v0 = smem_u32(sV), p0 = smem_u32(sP);
      bool ok = mbar_wait(&q_full, 0, &abort_flag);
      tc_fence_after_sync();
      for (int i = 0; ok && i <= n_blocks; ++i) {
        if (i < n_blocks) {
          const int st = i & 1, b = i & 1;
          if (!mbar_wait(&k_full[st], (i >> 1) & 1, &abort_flag)) break;
          if (i >= 2 && !mbar_wait(&s_free[b], ((i >> 1) + 1) & 1, &abort_flag)) break;
          tc_fence_after_sync();
          const uint32_t kb = k0 + st * L::kKV;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * L::kChunk + (kk & 3) * 32;
            umma_ss(tmem_s0 + b * kBlockN, smem_desc_sw128(q0 + off, 16, 1024), smem_desc_sw128(kb + off, 16, 1024),
                    kIdescS, kk > 0);
          }
          umma_commit(&s_full[b]);
          umma_commit(&k_empty[st]);
        }
        if (i >= 1) {
          const int j = i - 1, st = j & 1;
          if (!mbar_wait(&v_full[st], (j >> 1) & 1, &abort_flag)) break;
          if (!mbar_wait(&p_full, j & 1, &abort_flag)) break;
          tc_fence_after_sync();
          const uint32_t vb = v0 + st * L::kKV;
#pragma unroll
          for (int kk = 0; kk < kBlockN / 16; ++kk) {
            const uint32_t poff = (kk >> 2) * L::kChunk + (kk & 3) * 32;
            umma_ss(tmem_o, smem_desc_sw128(p0 + poff, 16, 1024),
                    smem_desc_sw128(vb + kk * 16 * 128, L::kChunk, 1024), kIdescO, (j > 0 || kk > 0));
          }
          umma_commit(&o_done);
          umma_commit(&v_empty[st]);
        }
      }
      umma_commit(&drain);
      mbar_wait_drain(&drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const long long grow = static_cast<long long>(tile) * kBlockM + r;
    const int lo = p.row_lo[grow];
    const int hi = p.row_hi[grow];
    const bool valid = (grow < p.t_local) && (lo <= hi);
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    float m = -INFINITY, l = 0.f;
    BlockCursor cur;
    cur.init(tile_iv, n_iv);
    bool ok = true;
    for (int i = 0; i < n_blocks; ++i) {
      // a block never reaches past its interval's end: the next interval may
      // start inside it, and its keys must be counted there only
      const int kstart = cur.start;
      const int kend = cur.end;
      cur.next();
      const int b = i & 1;
      if (!warp_wait(&s_full[b], (i >> 1) & 1, &abort_flag)) { ok = false; break; }
      tc_fence_after_sync();
      float s[kBlockN];
#pragma unroll
      for (int c = 0; c < kBlockN / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(tmem_s0 + lane_off + b * kBlockN + c * 32, rr);
        tmem_ld_wait(rr);
#pragma unroll
        for (int j = 0; j < 32; ++j) s[c * 32 + j] = __uint_as_float(rr[j]) * p.scale_log2;
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[b]);

      const int row_end = min(hi, kend);
      const bool full = (kstart >= ti.max_lo) && (kstart + kBlockN - 1 <= min(ti.min_hi, kend));
      if (!full) {
#pragma unroll
        for (int j = 0; j < kBlockN; ++j) {
          const int key = kstart + j;
          if (key < lo || key > row_end) s[j] = -INFINITY;
        }
      }
      float mx = s[0];
#pragma unroll
      for (int j = 1; j < kBlockN; ++j) mx = fmaxf(mx, s[j]);
      const float m_new = fmaxf(m, mx);
      const bool grow_o = (m != -INFINITY) && (m_new > m + kRescaleThreshold);
      float alpha = 1.f;
      if (m == -INFINITY) {
        m = m_new;  // nothing accumulated yet: O and l are exactly zero
      } else if (grow_o) {
        alpha = ex2(m - m_new);
        l *= alpha;
        m = m_new;
      }
      bool o_ready = false;
      if (__any_sync(0xffffffffu, grow_o)) {
        if (i > 0) {
          if (!warp_wait(&o_done, (i - 1) & 1, &abort_flag)) { ok = false; break; }
          tc_fence_after_sync();
          o_ready = true;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t rr[32];
            tmem_ld32(tmem_o + lane_off + c * 32, rr);
            tmem_ld_wait(rr);
#pragma unroll
            for (int j = 0; j < 32; ++j) rr[j] = __float_as_uint(__uint_as_float(rr[j]) * alpha);
            tmem_st32(tmem_o + lane_off + c * 32, rr);
          }
          tmem_st_wait();
        }
      }
      const float mref = (m == -INFINITY) ? 0.f : m;
      uint32_t pk[kBlockN / 2];
      float rs = 0.f;
#pragma unroll
      for (int j = 0; j < kBlockN / 2; ++j) {
        const float e0 = ex2(s[2 * j] - mref);
        const float e1 = ex2(s[2 * j + 1] - mref);
        rs += e0 + e1;
        pk[j] = pack_bf16x2(e0, e1);
      }
      l += rs;
      // the single P buffer is free once O += P_{i-1} V_{i-1} has completed
      if (i > 0 && !o_ready) {
        if (!warp_wait(&o_done, (i - 1) & 1, &abort_flag)) { ok = false; break; }
      }
#pragma unroll
      for (int u = 0; u < kBlockN / 8; ++u) {
        const int region = u >> 3, uu = u & 7;
        uint4* dst = reinterpret_cast<uint4*>(sP + region * L::kChunk + r * 128 + ((uu ^ (r & 7)) << 4));
        *dst = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full);
    }
    // ---------------------------------------------------------- epilogue
    if (ok && n_blocks > 0) ok = warp_wait(&o_done, (n_blocks - 1) & 1, &abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after_sync();
    if (ok) {
      const float inv = (valid && l > 0.f) ? 1.f / l : 0.f;
      __nv_bfloat16* orow = p.out + (grow * p.Hq + h) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t rr[32];
        if (n_blocks > 0) {
          tmem_ld32(tmem_o + lane_off + c * 32, rr);
          tmem_ld_wait(rr);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) rr[j] = 0u;
        }
        uint32_t ob[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          ob[j] = pack_bf16x2(__uint_as_float(rr[2 * j]) * inv, __uint_as_float(rr[2 * j + 1]) * inv);
        if (grow < p.t_local) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) dst[q4] = make_uint4(ob[4 * q4], ob[4 * q4 + 1], ob[4 * q4 + 2], ob[4 * q4 + 3]);
        }
      }
      if (grow < p.t_local)
        p.lse[static_cast<long long>(h) * p.t_local + grow] =
            (valid && l > 0.f) ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (abort_flag && threadIdx.x == 0) record_error(p.err, CPTHD_ERR_TIMEOUT, item);
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// [rows, heads, d] bf16 tensor, boxes of 64 columns x 1 head x 128 rows, 128-byte swizzle.
static bool make_rows_heads_map(EncodeTiledFn enc, CUtensorMap* m, const void* base, long long rows, int heads,
                                int d) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(heads) * d * 2};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
static int launch_attn(const void* q, const void* k, const void* v, long long t_local, long long T, int Hq, int Hkv,
                       float scale_log2, const AttnWorkspace& ws, long long ntiles, void* out, float* lse,
                       int32_t* err, cudaStream_t s) {
  EncodeTiledFn enc = get_encode_tiled();
  if (enc == nullptr) return CPTHD_ERR_CUDA;
  CUtensorMap mq, mk, mv;
  if (!make_rows_heads_map(enc, &mq, q, t_local, Hq, D) || !make_rows_heads_map(enc, &mk, k, T, Hkv, D) ||
      !make_rows_heads_map(enc, &mv, v, T, Hkv, D))
    return CPTHD_ERR_UNSUPPORTED;
  AttnParams p;
  p.row_lo = ws.row_lo;
  p.row_hi = ws.row_hi;
  p.tile_info = ws.tile_info;
  p.intervals = ws.intervals;
  p.order = ws.order;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.t_local = t_local;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.max_blocks = static_cast<int>((T + kBlockN - 1) / kBlockN + kBlockM);
  p.scale_log2 = scale_log2;
  p.err = err;
  const int smem = AttnSmem<D>::kLaunchBytes;
  CPTHD_TRY_CUDA(cudaFuncSetAttribute(attn_fwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  const long long items = ntiles * Hq;
  if (items > INT32_MAX) return CPTHD_ERR_UNSUPPORTED;
  attn_fwd_tc_kernel<D><<<static_cast<unsigned>(items), kAttnThreads, smem, s>>>(mq, mk, mv, p);
  CPTHD_TRY_CUDA(cudaGetLastError());
  return CPTHD_OK;
}

}  // namespace cpthd

extern "C" int thd_causal_attn_workspace_size(int64_t t_local, int Hq, int Hkv, int d, size_t* bytes_host) {
  if (bytes_host == nullptr || t_local < 0 || Hq < 1 || Hkv < 1) return CPTHD_ERR_INVALID_ARG;
  (void)d;
  const long long ntiles = (t_local + cpthd::kBlockM - 1) / cpthd::kBlockM;
  *bytes_host = cpthd::attn_workspace_bytes(ntiles);
  return CPTHD_OK;
}

extern "C" int thd_causal_attn_fwd(const int32_t* q_slice_idx_dev, int64_t t_local, const void* q_dev,
                                   const void* k_dev, const void* v_dev, int64_t T,
                                   const int32_t* cu_seqlens_dev, const int32_t* cu_seqlens_padded_dev,
                                   int num_docs, int Hq, int Hkv, int d, float softmax_scale, void* out_dev,
                                   float* lse_dev, void* workspace_dev, size_t workspace_bytes,
                                   int32_t* err_dev, cpthd_stream_t stream) {
  using namespace cpthd;
  if (t_local < 0 || T < 0 || T > INT32_MAX || t_local > INT32_MAX || num_docs < 0 || Hq < 1 || Hkv < 1)
    return CPTHD_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return CPTHD_ERR_UNSUPPORTED;
  if (Hq % Hkv != 0 || Hq > 65535) return CPTHD_ERR_UNSUPPORTED;
  if (t_local == 0) return CPTHD_OK;
  if (q_slice_idx_dev == nullptr || q_dev == nullptr || k_dev == nullptr || v_dev == nullptr ||
      cu_seqlens_dev == nullptr || out_dev == nullptr || lse_dev == nullptr || num_docs < 1 || T < 1)
    return CPTHD_ERR_INVALID_ARG;
  const uintptr_t align = reinterpret_cast<uintptr_t>(q_dev) | reinterpret_cast<uintptr_t>(k_dev) |
                          reinterpret_cast<uintptr_t>(v_dev) | reinterpret_cast<uintptr_t>(out_dev);
  if (align & 15) return CPTHD_ERR_UNSUPPORTED;
  const long long ntiles = (t_local + kBlockM - 1) / kBlockM;
  if (workspace_dev == nullptr || workspace_bytes < attn_workspace_bytes(ntiles) ||
      (reinterpret_cast<uintptr_t>(workspace_dev) & 255))
    return CPTHD_ERR_WORKSPACE;
  const int32_t* cup = cu_seqlens_padded_dev ? cu_seqlens_padded_dev : cu_seqlens_dev;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf(static_cast<float>(d));
  const float scale_log2 = scale * 1.4426950408889634f;

  AttnWorkspace ws = carve_workspace(workspace_dev, ntiles);
  attn_validate_docs_kernel<<<grid_for(num_docs + 1, 256, 64), 256, 0, s>>>(cu_seqlens_dev, cup, num_docs, T,
                                                                            err_dev);
  attn_tile_meta_kernel<<<static_cast<unsigned>(ntiles), kBlockM, 0, s>>>(
      q_slice_idx_dev, t_local, cu_seqlens_dev, cup, num_docs, T, ws, err_dev);
  attn_tile_order_kernel<<<1, 1024, 0, s>>>(static_cast<int>(ntiles), ws);
  CPTHD_TRY_CUDA(cudaGetLastError());
  if (d == 128) return launch_attn<128>(q_dev, k_dev, v_dev, t_local, T, Hq, Hkv, scale_log2, ws, ntiles, out_dev,
                                        lse_dev, err_dev, s);
  return launch_attn<64>(q_dev, k_dev, v_dev, t_local, T, Hq, Hkv, scale_log2, ws, ntiles, out_dev, lse_dev,
                         err_dev, s);
}
