// Pieces shared by the attention forward and backward kernels: the key-block
// cursor over a tile's intervals, bounded warp-uniform waits, and the TMA
// tensor maps of [rows, heads, d] bf16 tensors.
#pragma once

#include <cuda_bf16.h>

#include "attn_meta.cuh"
#include "common.cuh"
#include "sm100.cuh"

namespace cpthd {

using namespace sm100;

// Walks the key blocks of a group: interval by interval, 128 keys at a time.
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
  // Moves on by nb blocks (whole intervals at a time, then within one).
  __device__ void skip(int nb) {
    while (nb > 0 && k < n_iv) {
      const int left = (end >= start) ? (end - start) / kBlockN + 1 : 0;  // blocks left in this interval
      if (nb < left) {
        start += nb * kBlockN;
        return;
      }
      nb -= left;
      if (++k < n_iv) { int2 a = iv[k]; start = a.x; end = a.y; }
    }
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

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static inline EncodeTiledFn get_encode_tiled() {
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

// [rows, heads, d] bf16 tensor, boxes of 64 columns x 1 head x box_rows rows, 128-byte swizzle.
static inline bool make_rows_heads_map(EncodeTiledFn enc, CUtensorMap* m, const void* base, long long rows, int heads,
                                int d, int box_rows = 128) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(heads) * d * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Host checks of the scalar shape arguments shared by the forward entry
// points (the workspace and static-scratch forms run the same checks in the
// same order).
static inline int check_attn_shape(int64_t t_local, int64_t T, int num_docs, int Hq, int Hkv) {
  if (t_local < 0 || T < 0 || T > INT32_MAX || t_local > INT32_MAX || num_docs < 0 || Hq < 1 || Hkv < 1)
    return CPTHD_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || Hq > 65535) return CPTHD_ERR_UNSUPPORTED;
  return CPTHD_OK;
}

// Two query tiles per CTA: two heads of one KV head when the GQA group size is
// even, else two consecutive 128-row tiles of one head.
static inline int group_rows_for(int Hq, int Hkv) { return ((Hq / Hkv) % 2 == 0) ? kBlockM : 2 * kBlockM; }


}  // namespace cpthd
