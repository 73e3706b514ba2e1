// Causal packed-THD attention backward (dQ, dK, dV) on tcgen05 (sm_103a).
//
// The backward of the forward in attn_fwd.cu, for one context-parallel rank:
// the rank's query slice against the full K/V buffer, with the layout and the
// LSE the forward produced (TransformerEngine PR #3221: the strategy is
// captured for backward so forward and backward use the same token layout).
// With P = exp(scale q.k - lse) over the allowed pairs and D = rowsum(dO * O):
//   dV_k += P dO_q,   dS = P (dO_q . v_k - D_q),
//   dQ_q += scale dS k_k,   dK_k += scale dS q_q.
// dK and dV cover the whole [T, Hkv, d] buffer and hold this rank's
// contribution (what a reduce-scatter across CP ranks would sum); K/V heads
// collect every query head of their GQA group.
//
// No atomics: two passes, each owning its outputs.
//  * dQ pass, one CTA per (128-row query tile, query head), walking the
//    tile's key blocks exactly as the forward does: S = Q K^T and
//    dP = dO V^T into TMEM, the elementwise warps turn them into dS (bf16,
//    written back over S), then dQ += dS K with dS read from TMEM. Two S
//    buffers let S(j+1) and dQ(j) run while the elementwise warps work.
//  * dK/dV pass, persistent: one CTA per SM takes (128-key tile, KV head)
//    items from a counter; an item runs over every query tile whose key
//    intervals reach the key tile and every query head of the group (keys no
//    query reaches get zeros, so dK/dV need no clearing pass): S^T = K Q^T
//    and dP^T = V dO^T into TMEM, each with one more K step that subtracts
//    the per-query term (lse2 / (scale log2(e)), resp. D: a ones operand
//    times a per-query operand the pre-pass writes), the elementwise warps
//    write P^T and then dS^T (bf16) back over them in two phases, and
//    dV += P^T dO and dK += dS^T Q, both accumulated in TMEM and written
//    once per item, run during the other phase. With the per-query terms in
//    the scores, the elementwise loops read no shared memory (the SS-form
//    MMAs keep its bandwidth busy).
// The dK/dV pass reads nothing the dQ pass writes: it is launched as a
// programmatic dependent of the dQ pass and starts once every dQ CTA has
// started, taking the SMs the dQ pass's last wave leaves idle; it waits for
// the dQ grid only before it exits.
// Rows without keys get lse2 = +inf in the pre-pass (p = 0 without a mask);
// blocks and items the query tile's bounds cover fully skip the mask.
// Warp roles as in the forward: warp 0 TMA producer, warp 1 MMA issuer
// (owns TMEM), warps 2-5 elementwise (thread = TMEM lane). Every wait is
// bounded; a timeout drains, frees TMEM and records CPTHD_ERR_TIMEOUT.
#include "attn_common.cuh"

namespace cpthd {

constexpr int kBwdThreads = 192;
constexpr int kBwdMaxTiles = 2048;  // query tiles of one slice the dK/dV pass can list
// The dK/dV pass lets the tensor core add the per-query terms of
// x = s scale log2(e) - lse2 and of dP - D: one more K = 16 step of S^T and of
// dP^T multiplies a "ones" operand (128 keys x 16, ones in columns 0-2) by a
// per-query operand (128 queries x 16) that holds -lse2 / (scale log2(e)),
// resp. -D, as the sum of three bf16 terms in columns 0-2 (about 24
// significant bits). Both are K-major without swizzle: core matrices of 8
// rows x 16 bytes, row group g and K half c at byte g * 256 + c * 128.
constexpr int kBwdAugOperand = kBlockM * 16 * 2;     // one 128 x 16 bf16 operand
constexpr int kBwdAugBytes = 2 * kBwdAugOperand;     // per (query tile, head): the lse2 terms, then the D terms
constexpr int kBwdOnesBytes = kBlockN * 16 * 2;

template <int D>
struct BwdSmem {
  static constexpr int kChunk = kBlockM * 64 * 2;
  static constexpr int kChunks = D / 64;
  static constexpr int kTile = kChunks * kChunk;  // one 128-row bf16 tile of Q, dO, K or V
  static constexpr int kCol = 2 * kBlockM * 4;    // row_lo, row_hi of 128 query rows
  // dQ pass: Q, dO, K[3], V[2]
  static constexpr int kDqBytes = 7 * kTile;
  // dK/dV pass: K, V, Q[2], dO[2], column terms[2], the ones operand,
  // row bounds[2], two tile lists
  static constexpr int kDkvBytes = 6 * kTile + 2 * kBwdAugBytes + kBwdOnesBytes + 2 * kCol + 2 * kBwdMaxTiles * 2;
  static constexpr int launch(int b) { return (b + 1024 > 120 * 1024) ? b + 1024 : 120 * 1024; }
};

struct BwdParams {
  const int32_t* row_lo;
  const int32_t* row_hi;
  const GroupInfo* tile_info;
  const int2* intervals;
  const int32_t* order;  // dQ grid: query tiles by decreasing block count; null = natural order
  const float* lse2;  // [Hq, rows_pad]: lse * log2(e)
  const float* dvec;  // [Hq, rows_pad]: rowsum(dO * O)
  const uint8_t* aug;  // [Hq, ntiles] blocks of kBwdAugBytes: the dK/dV pass's per-query MMA operands
  float* dq;
  float* dk;
  float* dv;
  int32_t* work;  // dK/dV pass: [0] next work item (cleared by the pre-pass)
  long long t_local;
  long long T;
  int Hq;
  int Hkv;
  int ntiles;
  int n_key_tiles;
  int rows_pad;
  int max_blocks;
  float scale;
  float scale_log2;
  int32_t* err;
};

// Three bf16 terms whose sum is v to about 24 significant bits, in the low
// halves of a (element 0), then b (element 1), c (element 2).
__device__ __forceinline__ void split_bf16x3(float v, uint32_t& w01, uint32_t& w2) {
  const __nv_bfloat16 t0 = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(t0);
  const __nv_bfloat16 t1 = __float2bfloat16_rn(r1);
  const __nv_bfloat16 t2 = __float2bfloat16_rn(r1 - __bfloat162float(t1));
  w01 = static_cast<uint32_t>(__bfloat16_as_ushort(t0)) | (static_cast<uint32_t>(__bfloat16_as_ushort(t1)) << 16);
  w2 = static_cast<uint32_t>(__bfloat16_as_ushort(t2));
}

// D = rowsum(dO * O) and lse * log2(e), laid out [Hq, rows_pad]; one warp per (row, head).
// A row with no key (a pad row, LSE = -inf) or past the slice gets +inf, so
// that 2^(s*scale*log2(e) - lse2) is exactly 0 for it without any mask.
// Also the row's entries of the dK/dV pass's per-query operands: -lse2 /
// (scale log2(e)) (-2^120 for a row without keys, so that its scores end far
// below any exponent that ex2 keeps) and -D, each split into three bf16 terms.
template <int D>
static __global__ void __launch_bounds__(256) attn_bwd_pre_kernel(const __nv_bfloat16* __restrict__ out,
                                                                  const __nv_bfloat16* __restrict__ dout,
                                                                  const float* __restrict__ lse, long long t_local,
                                                                  int Hq, int rows_pad, float scale_log2, float* lse2,
                                                                  float* dvec, uint8_t* aug, int32_t* work) {
  if (blockIdx.x == 0 && threadIdx.x == 0) work[0] = 0;  // the dK/dV pass's work counter
  const long long w = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= (long long)rows_pad * Hq) return;
  const long long row = w / Hq;
  const int h = static_cast<int>(w - row * Hq);
  float acc = 0.f, l2 = INFINITY;
  if (row < t_local) {
    const __nv_bfloat16* o = out + (row * Hq + h) * D;
    const __nv_bfloat16* g = dout + (row * Hq + h) * D;
#pragma unroll
    for (int e = lane; e < D; e += 32) acc = fmaf(__bfloat162float(o[e]), __bfloat162float(g[e]), acc);
    const float l = lse[(long long)h * t_local + row];
    l2 = (l == -INFINITY) ? INFINITY : l * 1.4426950408889634f;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) {
    dvec[(long long)h * rows_pad + row] = acc;
    lse2[(long long)h * rows_pad + row] = l2;
  }
  if (lane < 2) {
    const float val = (lane == 1) ? -acc : (l2 == INFINITY ? -0x1p120f : -l2 / scale_log2);
    uint32_t w01, w2;
    split_bf16x3(val, w01, w2);
    const int ntiles = rows_pad / kBlockM, rr = static_cast<int>(row % kBlockM);
    uint8_t* blk = aug + (static_cast<long long>(h) * ntiles + row / kBlockM) * kBwdAugBytes + lane * kBwdAugOperand;
    uint4* dst = reinterpret_cast<uint4*>(blk + (rr >> 3) * 256 + (rr & 7) * 16);
    dst[0] = make_uint4(w01, w2, 0u, 0u);  // elements 0-7 of the row
    dst[8] = make_uint4(0u, 0u, 0u, 0u);    // elements 8-15, one core matrix further along K
  }
}

__device__ __forceinline__ void umma_desc_words(uint64_t d, uint32_t& lo, uint32_t& hi) {
  lo = static_cast<uint32_t>(d);
  hi = static_cast<uint32_t>(d >> 32);
}

// ------------------------------------------------------------------ dQ pass
// Software-pipelined over key blocks. TMEM holds two score buffers (S_0,
// S_1), dP and the dQ accumulator, so S(j+1) is computed while the
// elementwise warps turn block j into dS, and dP(j+1) is issued before
// dQ(j) += dS(j) K(j), so the next block's elementwise work overlaps dQ(j).
// K is held until dQ(j) and rides a three-stage ring; V, read by dP(j) only,
// a two-stage ring.
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const BwdParams p) {
  using L = BwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sDO = smem + L::kTile;
  uint8_t* sK = smem + 2 * L::kTile;  // three stages
  uint8_t* sV = smem + 5 * L::kTile;  // two stages

  __shared__ uint64_t qdo_full, k_full[3], k_empty[3], v_full[2], v_empty[2], sdp_full, ds_full, dq_final, drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  // The dK/dV pass depends on none of this pass's results: it may start as
  // soon as every CTA of this grid has started, and fill the SMs this grid's
  // last wave leaves idle.
  grid_dependents_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // with more CTAs than SMs the costliest query tiles go first
  const int tile = p.order ? __ldg(p.order + blockIdx.x / p.Hq) : static_cast<int>(blockIdx.x / p.Hq);
  const int h = blockIdx.x % p.Hq;
  const int kvh = h / (p.Hq / p.Hkv);
  const GroupInfo ti = p.tile_info[tile];
  const int n_blocks = min(max(ti.n_blocks, 0), p.max_blocks);
  const int2* tile_iv = p.intervals + static_cast<long long>(tile) * kBlockM;
  const int n_iv = min(max(ti.n_intervals, 0), kBlockM);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&qdo_full, 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(&sdp_full, 1);
    mbar_init(&ds_full, 4);
    mbar_init(&dq_final, 1);
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
  const uint32_t tmem = tmem_base_sh;  // S_0 [0,128), dP [128,256), dQ [256, 256+D), S_1 [384, 512)

  if (warp == 0) {
    if (lane == 0 && n_blocks > 0) {
      mbar_arrive_expect_tx(&qdo_full, 2 * L::kTile);
      for (int c = 0; c < L::kChunks; ++c) {
        tma_load_3d(sQ + c * L::kChunk, &tm_q, &qdo_full, c * 64, h, tile * kBlockM);
        tma_load_3d(sDO + c * L::kChunk, &tm_do, &qdo_full, c * 64, h, tile * kBlockM);
      }
      BlockCursor cur;
      cur.init(tile_iv, n_iv);
      int k_issued = 0, v_issued = 0;
      for (int i = 0; i < n_blocks; ++i) {
        // K(i) reuses the stage of K(i-3) (released by dQ(i-3)); V(i) that
        // of V(i-2) (released by dP(i-2)). Each release completes only
        // after loads issued here, so no wait runs two phases behind.
        const int ks = i % 3, vs = i & 1;
        if (i >= 3 && !mbar_wait(&k_empty[ks], ((i / 3) + 1) & 1, &abort_flag)) break;
        mbar_arrive_expect_tx(&k_full[ks], L::kTile);
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(sK + ks * L::kTile + c * L::kChunk, &tm_k, &k_full[ks], c * 64, kvh, cur.start);
        k_issued = i + 1;
        if (i >= 2 && !mbar_wait(&v_empty[vs], ((i >> 1) + 1) & 1, &abort_flag)) break;
        mbar_arrive_expect_tx(&v_full[vs], L::kTile);
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(sV + vs * L::kTile + c * L::kChunk, &tm_v, &v_full[vs], c * 64, kvh, cur.start);
        v_issued = i + 1;
        cur.next();
      }
      if (abort_flag) {
        // let every copy still in flight land before the CTA exits
        mbar_wait_drain(&qdo_full, 0);
        for (int i = (k_issued > 3 ? k_issued - 3 : 0); i < k_issued; ++i) mbar_wait_drain(&k_full[i % 3], (i / 3) & 1);
        for (int i = (v_issued > 2 ? v_issued - 2 : 0); i < v_issued; ++i) mbar_wait_drain(&v_full[i & 1], (i >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && n_blocks > 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(kBlockM, kBlockN, 0, 0);
      constexpr uint32_t kIdQ = idesc_bf16_f32(kBlockM, D, 0, 1);
      uint32_t q_lo, q_hi, do_lo, do_hi, k_lo, k_hi, kmn_lo, kmn_hi, v_lo, v_hi;
      umma_desc_words(smem_desc_sw128(smem_u32(sQ), 16, 1024), q_lo, q_hi);
      umma_desc_words(smem_desc_sw128(smem_u32(sDO), 16, 1024), do_lo, do_hi);
      umma_desc_words(smem_desc_sw128(smem_u32(sK), 16, 1024), k_lo, k_hi);
      umma_desc_words(smem_desc_sw128(smem_u32(sK), L::kChunk, 1024), kmn_lo, kmn_hi);
      umma_desc_words(smem_desc_sw128(smem_u32(sV), 16, 1024), v_lo, v_hi);
      auto t_sbuf = [&](int j) { return tmem + ((j & 1) ? 384u : 0u); };
      auto issue_s = [&](int j) {  // S(j) = Q K(j)^T into S_(j&1)
        const uint32_t so = ((j % 3) * L::kTile) >> 4;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * L::kChunk + (kk & 3) * 32) >> 4;
          umma_ss_w(t_sbuf(j), q_lo + off, q_hi, k_lo + so + off, k_hi, kIdS, kk > 0);
        }
      };
      auto issue_dp = [&](int j) {  // dP(j) = dO V(j)^T
        const uint32_t so = ((j & 1) * L::kTile) >> 4;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * L::kChunk + (kk & 3) * 32) >> 4;
          umma_ss_w(tmem + 128, do_lo + off, do_hi, v_lo + so + off, v_hi, kIdS, kk > 0);
        }
      };
      bool ok = mbar_wait(&qdo_full, 0, &abort_flag) && mbar_wait(&k_full[0], 0, &abort_flag) &&
                mbar_wait(&v_full[0], 0, &abort_flag);
      if (ok) {
        tc_fence_after_sync();
        issue_s(0);
        issue_dp(0);
        umma_commit(&sdp_full);
        umma_commit(&v_empty[0]);
      }
      for (int j = 0; ok && j < n_blocks; ++j) {
        const bool more = (j + 1 < n_blocks);
        if (more) {  // S(j+1) while the elementwise warps work on block j
          if (!mbar_wait(&k_full[(j + 1) % 3], ((j + 1) / 3) & 1, &abort_flag)) break;
          tc_fence_after_sync();
          issue_s(j + 1);
        }
        // dS(j) is in S_(j&1) and dP(j) has been read
        if (!mbar_wait(&ds_full, j & 1, &abort_flag)) break;
        tc_fence_after_sync();
        if (more) {
          if (!mbar_wait(&v_full[(j + 1) & 1], ((j + 1) >> 1) & 1, &abort_flag)) break;
          tc_fence_after_sync();
          issue_dp(j + 1);
          umma_commit(&sdp_full);  // reports S(j+1) and dP(j+1)
          umma_commit(&v_empty[(j + 1) & 1]);
        }
        const uint32_t acc0 = (j > 0) ? 1u : 0u;
        const uint32_t ko = ((j % 3) * L::kTile) >> 4;
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)  // dQ += dS K, dS from TMEM, K as the MN-major operand
          umma_ts_w(tmem + 256, t_sbuf(j) + kk * 8, kmn_lo + ko + ((kk * 16 * 128) >> 4), kmn_hi, kIdQ,
                    kk > 0 ? 1u : acc0);
        umma_commit(&k_empty[j % 3]);
      }
      umma_commit(&dq_final);
      umma_commit(&drain);
      mbar_wait_drain(&drain, 0);
    }
  } else {
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const long long grow = static_cast<long long>(tile) * kBlockM + r;
    const int lo = p.row_lo[grow], hi = p.row_hi[grow];
    const float lse2 = p.lse2[(long long)h * p.rows_pad + grow];
    const float drow = p.dvec[(long long)h * p.rows_pad + grow];
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_dp = tmem + lane_off + 128, t_q = tmem + lane_off + 256;
    const float sl2 = p.scale_log2;
    const int tmax_lo = ti.max_lo[0], tmin_hi = ti.min_hi[0];
    BlockCursor cur;
    cur.init(tile_iv, n_iv);
    bool ok = true;
    for (int j = 0; j < n_blocks; ++j) {
      const int kstart = cur.start, kend = cur.end;
      cur.next();
      if (!warp_wait(&sdp_full, j & 1, &abort_flag)) { ok = false; break; }
      tc_fence_after_sync();
      const uint32_t t_s = tmem + lane_off + ((j & 1) ? 384u : 0u);
      // allowed columns [c_lo, c_hi]; a pad row gets an empty range. A block
      // inside every real row's key interval needs no mask (a row without
      // keys has lse2 = +inf, so its p are 0 anyway).
      const bool full = (kstart >= tmax_lo) && (kstart + kBlockN - 1 <= min(tmin_hi, kend));
      const int c_lo = min(max(lo - kstart, 0), kBlockN);
      const int c_hi = max(min(min(hi, kend) - kstart, kBlockN - 1), -1);
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {  // 64 columns per load round trip
        uint32_t sv[64], dp[64];
        tmem_ld64(t_s + 64 * c2, sv);
        tmem_ld64(t_dp + 64 * c2, dp);
        tmem_ld_wait64(sv);
        tmem_ld_wait64(dp);
        uint32_t pk[32];
        if (full) {
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            // packed pairs: the same roundings as the scalar fma, sub and mul
            float a0, a1, t0, t1, d0, d1;
            fma2(a0, a1, __uint_as_float(sv[2 * q]), __uint_as_float(sv[2 * q + 1]), sl2, -lse2);
            fma2(t0, t1, __uint_as_float(dp[2 * q]), __uint_as_float(dp[2 * q + 1]), 1.f, -drow);
            mul2(d0, d1, ex2(a0), ex2(a1), t0, t1);
            pk[q] = pack_bf16x2(d0, d1);
          }
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            float ds2[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int col = 64 * c2 + 2 * q + u;
              const float e = ex2(fmaf(__uint_as_float(sv[2 * q + u]), sl2, -lse2));
              const float pv = (col >= c_lo && col <= c_hi) ? e : 0.f;
              ds2[u] = pv * (__uint_as_float(dp[2 * q + u]) - drow);
            }
            pk[q] = pack_bf16x2(ds2[0], ds2[1]);
          }
        }
        // dS over the first 64 S columns: columns 32 c2 .. 32 c2 + 31 hold
        // S values already read (this slab's or the previous one's)
        tmem_st32(t_s + 32 * c2, pk);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ds_full);
    }
    if (ok && n_blocks > 0) ok = warp_wait(&dq_final, 0, &abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after_sync();
    if (ok) {
      float* dst = p.dq + (grow * p.Hq + h) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t rr[32];
        if (n_blocks > 0) {
          tmem_ld32(t_q + 32 * c, rr);
          tmem_ld_wait(rr);
        }
        if (grow < p.t_local) {
          float4* d4 = reinterpret_cast<float4*>(dst + 32 * c);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float4 v;
            v.x = n_blocks > 0 ? __uint_as_float(rr[4 * q]) * p.scale : 0.f;
            v.y = n_blocks > 0 ? __uint_as_float(rr[4 * q + 1]) * p.scale : 0.f;
            v.z = n_blocks > 0 ? __uint_as_float(rr[4 * q + 2]) * p.scale : 0.f;
            v.w = n_blocks > 0 ? __uint_as_float(rr[4 * q + 3]) * p.scale : 0.f;
            d4[q] = v;
          }
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (abort_flag && threadIdx.x == 0) record_error(p.err, CPTHD_ERR_TIMEOUT, blockIdx.x);
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// --------------------------------------------------------------- dK/dV pass
// Persistent: one CTA per SM takes work items (128-key tile kt, KV head g):
// the first is its block index, the rest come from a counter (cleared by
// the pre-pass), claimed after the item's last Q/dO load. Work items run in
// key-tile order, the costliest first for causal slices (early keys are
// reached by the most query tiles).
// Roles: warp 0 builds each item's list of query tiles whose key intervals
// reach [kt*128, kt*128+127] (32 lanes with ballots, in tile order) into one
// of two list buffers and publishes the item; its lane 0 then loads K and V
// (once the previous item's last scores are issued: kv_empty) and the Q / dO
// tiles with their row data through a two-stage ring (numbered over all of
// the CTA's items). Warp 1 issues the MMAs; an item's first dV / dK MMA waits
// until the elementwise warps have read the previous item's dV / dK from TMEM
// (acc_free). Warps 2-5 run the elementwise phases and the epilogue; an item
// that no query reaches gets zeros.
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const BwdParams p) {
  using L = BwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = smem + L::kTile;
  uint8_t* sQ = smem + 2 * L::kTile;   // two stages
  uint8_t* sDO = smem + 4 * L::kTile;  // two stages
  uint8_t* sAug = smem + 6 * L::kTile;  // two stages of the per-query operands (lse2 terms, D terms)
  uint8_t* sOnes = sAug + 2 * kBwdAugBytes;
  uint8_t* sCol = sOnes + kBwdOnesBytes;  // two stages of {row_lo, row_hi} x 128
  // two lists of kBwdMaxTiles query tiles: the tile in bits 0-14, and bit 15
  // set when every real row of the tile sees all 128 keys
  uint16_t* sList = reinterpret_cast<uint16_t*>(sCol + 2 * L::kCol);

  __shared__ uint64_t kv_full, kv_empty, qdo_full[2], qdo_empty[2], sdp_full[2], pds_full[2], kv_final, acc_free;
  __shared__ uint64_t item_full[2], item_empty[2], drain;
  __shared__ int item_slot[2], list_n[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ int last_key_tile;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int group = p.Hq / p.Hkv;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&kv_full, 1);
    mbar_init(&kv_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&qdo_full[s], 1);
      mbar_init(&qdo_empty[s], 1);
      mbar_init(&sdp_full[s], 1);
      mbar_init(&pds_full[s], 4);
      mbar_init(&item_full[s], 1);
      mbar_init(&item_empty[s], 5);  // the MMA issuer and the four elementwise warps
    }
    mbar_init(&kv_final, 1);
    mbar_init(&acc_free, 4);
    mbar_init(&drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  // the ones operand: 1 in columns 0-2 of every row (the first core matrix
  // along K of each row group), 0 elsewhere
  for (int i = threadIdx.x; i < kBwdOnesBytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sOnes)[i] = ((i & 15) < 8) ? make_uint4(0x3f803f80u, 0x3f80u, 0u, 0u)
                                                        : make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // S^T [0,128), dP^T [128,256), dV [256,256+D), dK [256+D, 256+2D).
  const uint32_t tmem = tmem_base_sh;
  // the item's list length, from the published slot (items past the end: -1)
  auto items_of = [&](int slot) { return min(list_n[slot], kBwdMaxTiles) * group; };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The last key tile any query of the slice reaches (a tile's intervals
    // are sorted by document, so its last one ends at its largest slot):
    // work items stop there, and the tiles past it are zero-filled by the
    // whole grid after the item loop.
    int max_end = -1;
    for (int t = lane; t < p.ntiles; t += 32) {
      const int n_iv = min(max(p.tile_info[t].n_intervals, 0), kBlockM);
      if (n_iv > 0) max_end = max(max_end, min(p.intervals[static_cast<long long>(t) * kBlockM + n_iv - 1].y,
                                              static_cast<int>(p.T) - 1));
    }
    max_end = __reduce_max_sync(0xffffffffu, max_end);
    const int kt_last = (max_end < 0) ? -1 : max_end / kBlockN;
    if (lane == 0) last_key_tile = kt_last;
    const int n_work = (kt_last + 1) * p.Hkv;
    int next = blockIdx.x;
    int ig = 0;   // Q/dO items loaded so far, over all work items
    int nkv = 0;  // K/V loads so far
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int slot = k & 1;
      if (k >= 2) {
        bool w = true;
        if (lane == 0) w = mbar_wait(&item_empty[slot], ((k >> 1) - 1) & 1, &abort_flag);
        if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0)) break;
      }
      const int item = (next < n_work) ? next : -1;
      int count = 0;
      if (item >= 0) {
        // query tiles whose key intervals reach this key tile, in tile order
        const int K0 = (item / p.Hkv) * kBlockN;
        for (int base = 0; base < p.ntiles; base += 32) {
          const int t = base + lane;
          bool rel = false, full = false;
          if (t < p.ntiles) {
            const GroupInfo ti = p.tile_info[t];
            const int n_iv = min(max(ti.n_intervals, 0), kBlockM);
            const int2* iv = p.intervals + static_cast<long long>(t) * kBlockM;
            // the intervals are disjoint and in key order: the first start and
            // the last end bound them, which rejects most tiles at once
            if (n_iv > 0 && iv[0].x <= K0 + kBlockN - 1 && iv[n_iv - 1].y >= K0) {
              for (int q = 0; q < n_iv && !rel; ++q) {
                const int2 a = iv[q];
                rel = (a.x <= K0 + kBlockN - 1) && (a.y >= K0);
              }
            }
            full = (ti.max_lo[0] <= K0 && ti.min_hi[0] >= K0 + kBlockN - 1);
          }
          const unsigned ballot = __ballot_sync(0xffffffffu, rel);
          const int pos = count + __popc(ballot & ((1u << lane) - 1u));
          if (rel && pos < kBwdMaxTiles)
            sList[slot * kBwdMaxTiles + pos] = static_cast<uint16_t>(t | (full ? 0x8000 : 0));
          count += __popc(ballot);
        }
      }
      __threadfence_block();
      __syncwarp();
      if (lane == 0) {
        item_slot[slot] = item;
        list_n[slot] = count;
        mbar_arrive(&item_full[slot]);
      }
      if (item < 0) break;
      const int n_items = min(count, kBwdMaxTiles) * group;
      if (lane == 0 && n_items > 0) {
        const int kt = item / p.Hkv, g = item % p.Hkv;
        const int K0 = kt * kBlockN;
        // K and V of the previous item are read by its last S^T / dP^T
        if (nkv > 0 && !mbar_wait(&kv_empty, (nkv - 1) & 1, &abort_flag)) ok = false;
        if (ok) {
          mbar_arrive_expect_tx(&kv_full, 2 * L::kTile);
          for (int c = 0; c < L::kChunks; ++c) {
            tma_load_3d(sK + c * L::kChunk, &tm_k, &kv_full, c * 64, g, K0);
            tma_load_3d(sV + c * L::kChunk, &tm_v, &kv_full, c * 64, g, K0);
          }
          ++nkv;
        }
        for (int i = 0; ok && i < n_items; ++i, ++ig) {
          const int st = ig & 1;
          const int t = sList[slot * kBwdMaxTiles + i / group] & 0x7fff;
          const int h = g * group + i % group;
          // Q / dO stage st is free once dK of the item two before is done;
          // that barrier's next phase needs this load, so the parity is
          // unambiguous however far behind this thread runs
          if (ig >= 2 && !mbar_wait(&qdo_empty[st], ((ig >> 1) - 1) & 1, &abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&qdo_full[st], 2 * L::kTile + kBwdAugBytes + L::kCol);
          for (int c = 0; c < L::kChunks; ++c) {
            tma_load_3d(sQ + st * L::kTile + c * L::kChunk, &tm_q, &qdo_full[st], c * 64, h, t * kBlockM);
            tma_load_3d(sDO + st * L::kTile + c * L::kChunk, &tm_do, &qdo_full[st], c * 64, h, t * kBlockM);
          }
          uint8_t* col = sCol + st * L::kCol;
          const long long r0 = static_cast<long long>(t) * kBlockM;
          bulk_load(col, p.row_lo + r0, kBlockM * 4, &qdo_full[st]);
          bulk_load(col + kBlockM * 4, p.row_hi + r0, kBlockM * 4, &qdo_full[st]);
          bulk_load(sAug + st * kBwdAugBytes, p.aug + (static_cast<long long>(h) * p.ntiles + t) * kBwdAugBytes,
                    kBwdAugBytes, &qdo_full[st]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      ig = __shfl_sync(0xffffffffu, ig, 0);
      nkv = __shfl_sync(0xffffffffu, nkv, 0);
      // the next item is claimed once this one's loads are issued
      if (lane == 0) next = static_cast<int>(gridDim.x) + atomicAdd(p.work + 0, 1);
      next = __shfl_sync(0xffffffffu, next, 0);
    }
    if (lane == 0 && abort_flag) {
      // let every copy still in flight land before the CTA exits
      if (nkv > 0) mbar_wait_drain(&kv_full, (nkv - 1) & 1);
      for (int i = (ig > 2 ? ig - 2 : 0); i < ig; ++i) mbar_wait_drain(&qdo_full[i & 1], (i >> 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(kBlockM, kBlockN, 0, 0);
      constexpr uint32_t kIdO = idesc_bf16_f32(kBlockM, D, 0, 1);
      uint32_t k_lo, k_hi, v_lo, v_hi, q_lo, q_hi, do_lo, do_hi, qmn_lo, qmn_hi, domn_lo, domn_hi;
      umma_desc_words(smem_desc_sw128(smem_u32(sK), 16, 1024), k_lo, k_hi);
      umma_desc_words(smem_desc_sw128(smem_u32(sV), 16, 1024), v_lo, v_hi);
      umma_desc_words(smem_desc_sw128(smem_u32(sQ), 16, 1024), q_lo, q_hi);
      umma_desc_words(smem_desc_sw128(smem_u32(sDO), 16, 1024), do_lo, do_hi);
      umma_desc_words(smem_desc_sw128(smem_u32(sQ), L::kChunk, 1024), qmn_lo, qmn_hi);
      umma_desc_words(smem_desc_sw128(smem_u32(sDO), L::kChunk, 1024), domn_lo, domn_hi);
      uint32_t one_lo, one_hi, aug_lo, aug_hi;
      umma_desc_words(smem_desc_noswizzle(smem_u32(sOnes), 128, 256), one_lo, one_hi);
      umma_desc_words(smem_desc_noswizzle(smem_u32(sAug), 128, 256), aug_lo, aug_hi);
      auto issue_s = [&](int i) {  // S^T = K Q^T - lse2 / (scale log2(e)) into [0, 128)
        const uint32_t so = ((i & 1) * L::kTile) >> 4;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * L::kChunk + (kk & 3) * 32) >> 4;
          umma_ss_w(tmem, k_lo + off, k_hi, q_lo + so + off, q_hi, kIdS, kk > 0);
        }
        umma_ss_w(tmem, one_lo, one_hi, aug_lo + (((i & 1) * kBwdAugBytes) >> 4), aug_hi, kIdS, 1u);
      };
      auto issue_dp = [&](int i) {  // dP^T = V dO^T - D into [128, 256)
        const uint32_t so = ((i & 1) * L::kTile) >> 4;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * L::kChunk + (kk & 3) * 32) >> 4;
          umma_ss_w(tmem + 128, v_lo + off, v_hi, do_lo + so + off, do_hi, kIdS, kk > 0);
        }
        umma_ss_w(tmem + 128, one_lo, one_hi, aug_lo + (((i & 1) * kBwdAugBytes + kBwdAugOperand) >> 4), aug_hi, kIdS,
                  1u);
      };
      auto issue_dv = [&](int i, uint32_t acc0) {  // dV (+)= P^T dO, P^T (bf16) in [0, 64)
        const uint32_t so = ((i & 1) * L::kTile) >> 4;
#pragma unroll
        for (int kk = 0; kk < kBlockM / 16; ++kk)
          umma_ts_w(tmem + 256, tmem + kk * 8, domn_lo + so + ((kk * 16 * 128) >> 4), domn_hi, kIdO,
                    kk > 0 ? 1u : acc0);
      };
      auto issue_dk = [&](int i, uint32_t acc0) {  // dK (+)= dS^T Q, dS^T (bf16) in [128, 192)
        const uint32_t so = ((i & 1) * L::kTile) >> 4;
#pragma unroll
        for (int kk = 0; kk < kBlockM / 16; ++kk)
          umma_ts_w(tmem + 256 + D, tmem + 128 + kk * 8, qmn_lo + so + ((kk * 16 * 128) >> 4), qmn_hi, kIdO,
                    kk > 0 ? 1u : acc0);
      };
      int ig = 0, nkv = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int slot = k & 1;
        if (!mbar_wait(&item_full[slot], (k >> 1) & 1, &abort_flag)) break;
        const int item = item_slot[slot];
        const int n_items = items_of(slot);
        mbar_arrive(&item_empty[slot]);  // the issuer needs only the count
        if (item < 0) break;
        if (n_items == 0 && k > 0) {
          // no MMA, but this item's kv_final must not come before the
          // previous item's dV / dK have been read out of TMEM
          if (!mbar_wait(&acc_free, (k - 1) & 1, &abort_flag)) ok = false;
        }
        if (ok && n_items > 0) {
          ok = mbar_wait(&kv_full, nkv & 1, &abort_flag) && mbar_wait(&qdo_full[ig & 1], (ig >> 1) & 1, &abort_flag);
          ++nkv;
          if (ok) {
            tc_fence_after_sync();
            issue_s(ig);
            umma_commit(&sdp_full[0]);
            issue_dp(ig);
            umma_commit(&sdp_full[1]);
            if (n_items == 1) umma_commit(&kv_empty);  // the item's last reads of K and V are issued
          }
          for (int i = 0; ok && i < n_items; ++i) {
            const int gi = ig + i;
            const bool more = (i + 1 < n_items);
            // the previous item's dV / dK have been read out of TMEM before
            // this item's first dV / dK overwrite them
            if (i == 0 && k > 0 && !mbar_wait(&acc_free, (k - 1) & 1, &abort_flag)) { ok = false; break; }
            // phase 1 of item gi done: P^T(gi) in [0, 64)
            if (!mbar_wait(&pds_full[0], gi & 1, &abort_flag)) { ok = false; break; }
            tc_fence_after_sync();
            issue_dv(gi, i > 0 ? 1u : 0u);
            if (more) {  // S^T(gi+1) overwrites [0, 128) only after dV(gi) (issue order)
              if (!mbar_wait(&qdo_full[(gi + 1) & 1], ((gi + 1) >> 1) & 1, &abort_flag)) { ok = false; break; }
              tc_fence_after_sync();
              issue_s(gi + 1);
              umma_commit(&sdp_full[0]);
            }
            // phase 2 of item gi done: dS^T(gi) in [128, 192)
            if (!mbar_wait(&pds_full[1], gi & 1, &abort_flag)) { ok = false; break; }
            tc_fence_after_sync();
            issue_dk(gi, i > 0 ? 1u : 0u);
            umma_commit(&qdo_empty[gi & 1]);  // Q(gi), dO(gi) and their column data are free
            if (more) {  // dP^T(gi+1) overwrites [128, 256) only after dK(gi)
              issue_dp(gi + 1);
              umma_commit(&sdp_full[1]);
              if (i + 2 == n_items) umma_commit(&kv_empty);
            }
          }
          ig += n_items;
        }
        umma_commit(&kv_final);  // this item's dV / dK are complete (or it had none)
      }
      umma_commit(&drain);
      mbar_wait_drain(&drain, 0);
    }
  } else {
    // ------------------------------------------------------------ elementwise
    // One thread per key (TMEM lane), in two phases per query item: phase 1
    // turns S^T into P^T (bf16, over the first 64 columns of S^T) and keeps
    // P as bf16 pairs in registers; phase 2 turns dP^T into
    // dS^T = P (dP^T - D) (bf16, over the first 64 columns of dP^T). The
    // issuer runs dV(i) and S^T(i+1) during phase 2, and dK(i) and
    // dP^T(i+1) during the next phase 1.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_off, t_dp = tmem + lane_off + 128;
    const uint32_t t_v = tmem + lane_off + 256, t_k = tmem + lane_off + 256 + D;
    const float sl2 = p.scale_log2;
    int ig = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int slot = k & 1;
      if (!warp_wait(&item_full[slot], (k >> 1) & 1, &abort_flag)) break;
      const int item = item_slot[slot];
      if (item < 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&item_empty[slot]);
        break;
      }
      const int n_items = items_of(slot);
      const int kt = item / p.Hkv, g = item % p.Hkv;
      const int key = kt * kBlockN + r;
      for (int i = 0; ok && i < n_items; ++i) {
        const int gi = ig + i;
        const int st = gi & 1;
        // the column data arrived with Q/dO through the TMA barrier
        if (!warp_wait(&qdo_full[st], (gi >> 1) & 1, &abort_flag)) { ok = false; break; }
        const int* c_lo = reinterpret_cast<const int*>(sCol + st * L::kCol);
        const int* c_hi = c_lo + kBlockM;
        const bool item_full_keys = (sList[slot * kBwdMaxTiles + i / group] & 0x8000) != 0;
        uint32_t pp[64];  // P of the 128 queries, bf16 pairs
        // ---- phase 1: P = 2^(S scale log2(e) - lse2), masked; S^T already
        // holds S - lse2 / (scale log2(e)), so no per-query value is read here
        // (unless a mask is needed)
        if (!warp_wait(&sdp_full[0], gi & 1, &abort_flag)) { ok = false; break; }
        tc_fence_after_sync();
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          uint32_t sv[64];
          tmem_ld64(t_s + 64 * c2, sv);
          tmem_ld_wait64(sv);
#pragma unroll
          for (int q4 = 0; q4 < 16; ++q4) {
            const int col = 64 * c2 + 4 * q4;
            float pv[4];
#pragma unroll
            for (int u = 0; u < 4; u += 2) {
              float a0, a1;
              mul2(a0, a1, __uint_as_float(sv[4 * q4 + u]), __uint_as_float(sv[4 * q4 + u + 1]), sl2, sl2);
              pv[u] = ex2(a0);
              pv[u + 1] = ex2(a1);
            }
            if (!item_full_keys) {
              const int4 lo4 = *reinterpret_cast<const int4*>(c_lo + col);
              const int4 hi4 = *reinterpret_cast<const int4*>(c_hi + col);
              const int los[4] = {lo4.x, lo4.y, lo4.z, lo4.w};
              const int his[4] = {hi4.x, hi4.y, hi4.z, hi4.w};
#pragma unroll
              for (int u = 0; u < 4; ++u) pv[u] = (key >= los[u] && key <= his[u]) ? pv[u] : 0.f;
            }
            pp[32 * c2 + 2 * q4] = pack_bf16x2(pv[0], pv[1]);
            pp[32 * c2 + 2 * q4 + 1] = pack_bf16x2(pv[2], pv[3]);
          }
          // P^T of these 64 queries over columns 32 c2 .. 32 c2 + 31, already read
          uint32_t (&half)[32] = *reinterpret_cast<uint32_t(*)[32]>(pp + 32 * c2);
          tmem_st32(t_s + 32 * c2, half);
        }
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pds_full[0]);
        // ---- phase 2: dS = P (dP - D); dP^T already holds dP - D
        if (!warp_wait(&sdp_full[1], gi & 1, &abort_flag)) { ok = false; break; }
        tc_fence_after_sync();
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          uint32_t dp[64];
          tmem_ld64(t_dp + 64 * c2, dp);
          tmem_ld_wait64(dp);
          uint32_t pd[32];
#pragma unroll
          for (int q4 = 0; q4 < 16; ++q4) {
            const uint32_t w0 = pp[32 * c2 + 2 * q4], w1 = pp[32 * c2 + 2 * q4 + 1];
            const float pv[4] = {__uint_as_float(w0 << 16), __uint_as_float(w0 & 0xffff0000u),
                                 __uint_as_float(w1 << 16), __uint_as_float(w1 & 0xffff0000u)};
            float dsv[4];
#pragma unroll
            for (int u = 0; u < 4; u += 2)
              mul2(dsv[u], dsv[u + 1], pv[u], pv[u + 1], __uint_as_float(dp[4 * q4 + u]),
                   __uint_as_float(dp[4 * q4 + u + 1]));
            pd[2 * q4] = pack_bf16x2(dsv[0], dsv[1]);
            pd[2 * q4 + 1] = pack_bf16x2(dsv[2], dsv[3]);
          }
          tmem_st32(t_dp + 32 * c2, pd);  // dS^T over columns already read
        }
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pds_full[1]);
      }
      ig += n_items;
      // ---- epilogue: this key tile's dV and dK (zeros when no query reaches it)
      if (ok) ok = warp_wait(&kv_final, k & 1, &abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after_sync();
      float* dv_row = p.dv + (static_cast<long long>(key) * p.Hkv + g) * D;
      float* dk_row = p.dk + (static_cast<long long>(key) * p.Hkv + g) * D;
      if (ok && n_items > 0) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rv[32], rk[32];
          tmem_ld32(t_v + 32 * c, rv);
          tmem_ld32(t_k + 32 * c, rk);
          tmem_ld_wait(rv);
          tmem_ld_wait(rk);
          if (c == D / 32 - 1) {
            // dV / dK are in registers: the next item's first MMAs may overwrite them
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_free);
          }
          if (key < p.T) {
            float4* dv4 = reinterpret_cast<float4*>(dv_row + 32 * c);
            float4* dk4 = reinterpret_cast<float4*>(dk_row + 32 * c);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              dv4[q] = make_float4(__uint_as_float(rv[4 * q]), __uint_as_float(rv[4 * q + 1]),
                                   __uint_as_float(rv[4 * q + 2]), __uint_as_float(rv[4 * q + 3]));
              dk4[q] = make_float4(__uint_as_float(rk[4 * q]) * p.scale, __uint_as_float(rk[4 * q + 1]) * p.scale,
                                   __uint_as_float(rk[4 * q + 2]) * p.scale,
                                   __uint_as_float(rk[4 * q + 3]) * p.scale);
            }
          }
        }
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_free);
        if (ok && key < p.T) {
          // no query of the slice reaches these keys: their contribution is zero
          float4* dv4 = reinterpret_cast<float4*>(dv_row);
          float4* dk4 = reinterpret_cast<float4*>(dk_row);
#pragma unroll 8
          for (int q = 0; q < D / 4; ++q) {
            dv4[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            dk4[q] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[slot]);  // done with this item's list
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (abort_flag && threadIdx.x == 0) record_error(p.err, CPTHD_ERR_TIMEOUT, blockIdx.x);
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem, 512);
  // keys past the last reached key tile: zeros, spread over the whole grid
  const long long first = static_cast<long long>(last_key_tile + 1) * kBlockN;
  if (first < p.T) {
    const long long n4 = (p.T - first) * p.Hkv * D / 4;
    float4* dk4 = reinterpret_cast<float4*>(p.dk + first * p.Hkv * D);
    float4* dv4 = reinterpret_cast<float4*>(p.dv + first * p.Hkv * D);
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
      dk4[i] = z;
      dv4[i] = z;
    }
  }
  // This grid may have started beside the dQ pass (it reads nothing the dQ
  // pass writes); it ends only after that pass has, so that the backward
  // call's completion covers both.
  grid_dependency_wait();
}

static size_t bwd_workspace_bytes(long long ntiles, int Hq) {
  const long long rows_pad = ntiles * kBlockM;
  return attn_workspace_bytes(ntiles, kBlockM) + 2 * align256(sizeof(float) * rows_pad * Hq) +
         align256(sizeof(int32_t) * 8) + align256(static_cast<size_t>(kBwdAugBytes) * ntiles * Hq);
}

template <int D>
static int launch_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
                      const float* lse, long long t_local, long long T, int Hq, int Hkv, float scale,
                      const AttnWorkspace& ws, float* lse2, float* dvec, uint8_t* aug, int32_t* work, long long ntiles,
                      float* dq,
                      float* dk, float* dv, int32_t* err, cudaStream_t s) {
  EncodeTiledFn enc = get_encode_tiled();
  if (enc == nullptr) return CPTHD_ERR_CUDA;
  CUtensorMap mq, mdo, mk, mv;
  if (!make_rows_heads_map(enc, &mq, q, t_local, Hq, D) || !make_rows_heads_map(enc, &mdo, dout, t_local, Hq, D) ||
      !make_rows_heads_map(enc, &mk, k, T, Hkv, D) || !make_rows_heads_map(enc, &mv, v, T, Hkv, D))
    return CPTHD_ERR_UNSUPPORTED;
  const int rows_pad = static_cast<int>(ntiles * kBlockM);
  const long long warps = static_cast<long long>(rows_pad) * Hq;
  attn_bwd_pre_kernel<D><<<static_cast<unsigned>((warps + 7) / 8), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), lse, t_local, Hq, rows_pad,
      scale * 1.4426950408889634f, lse2, dvec, aug, work);
  // The dQ grid runs in decreasing-cost order (the forward's group order
  // over the query tiles) when it needs more than one wave of CTAs.
  const bool ordered = ntiles * Hq > sm_count();
  if (ordered)
    attn_group_order_kernel<<<1, 1024, 0, s>>>(static_cast<int>(ntiles), &ws.group_info[0].n_blocks,
                                               static_cast<int>(sizeof(GroupInfo) / sizeof(int)), ws.order);
  BwdParams p;
  p.row_lo = ws.row_lo;
  p.row_hi = ws.row_hi;
  p.tile_info = ws.group_info;
  p.intervals = ws.intervals;
  p.order = ordered ? ws.order : nullptr;
  p.lse2 = lse2;
  p.dvec = dvec;
  p.aug = aug;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.work = work;
  p.t_local = t_local;
  p.T = T;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.ntiles = static_cast<int>(ntiles);
  p.n_key_tiles = static_cast<int>((T + kBlockN - 1) / kBlockN);
  p.rows_pad = rows_pad;
  p.max_blocks = static_cast<int>((T + kBlockN - 1) / kBlockN + kBlockM);
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.err = err;
  const int smem_dq = BwdSmem<D>::launch(BwdSmem<D>::kDqBytes);
  const int smem_kv = BwdSmem<D>::launch(BwdSmem<D>::kDkvBytes);
  CPTHD_TRY_CUDA(cudaFuncSetAttribute(attn_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_dq));
  CPTHD_TRY_CUDA(cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_kv));
  attn_bwd_dq_kernel<D><<<static_cast<unsigned>(ntiles * Hq), kBwdThreads, smem_dq, s>>>(mq, mdo, mk, mv, p);
  // persistent: one CTA per SM, taking (key tile, KV head) items
  const long long work_items = static_cast<long long>(p.n_key_tiles) * Hkv;
  const int sms = sm_count();
  if (sms < 1) return CPTHD_ERR_CUDA;
  const long long grid_kv = work_items < sms ? work_items : sms;
  // launched to overlap the dQ pass's last wave (see the two kernels)
  CPTHD_TRY_CUDA(cudaGetLastError());
  CPTHD_TRY_CUDA(launch_pdl(attn_bwd_dkdv_kernel<D>, dim3(static_cast<unsigned>(grid_kv)), dim3(kBwdThreads),
                            static_cast<size_t>(smem_kv), s, mq, mdo, mk, mv, p));
  return CPTHD_OK;
}

}  // namespace cpthd

extern "C" int thd_causal_attn_bwd_workspace_size(int64_t t_local, int Hq, int Hkv, int d, size_t* bytes_host) {
  if (bytes_host == nullptr || t_local < 0 || Hq < 1 || Hkv < 1) return CPTHD_ERR_INVALID_ARG;
  (void)Hkv;
  (void)d;
  const long long ntiles = (t_local + cpthd::kBlockM - 1) / cpthd::kBlockM;
  *bytes_host = cpthd::bwd_workspace_bytes(ntiles, Hq);
  return CPTHD_OK;
}

extern "C" int thd_causal_attn_bwd(const int32_t* q_slice_idx_dev, int64_t t_local, const void* q_dev,
                                   const void* k_dev, const void* v_dev, const void* out_dev, const void* dout_dev,
                                   const float* lse_dev, int64_t T, const int32_t* cu_seqlens_dev,
                                   const int32_t* cu_seqlens_padded_dev, int num_docs, int Hq, int Hkv, int d,
                                   float softmax_scale, float* dq_dev, float* dk_dev, float* dv_dev,
                                   void* workspace_dev, size_t workspace_bytes, int32_t* err_dev,
                                   cpthd_stream_t stream) {
  using namespace cpthd;
  if (t_local < 0 || T < 0 || T > INT32_MAX || t_local > INT32_MAX || num_docs < 0 || Hq < 1 || Hkv < 1)
    return CPTHD_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return CPTHD_ERR_UNSUPPORTED;
  if (Hq % Hkv != 0 || Hq > 65535) return CPTHD_ERR_UNSUPPORTED;
  const long long ntiles = (t_local + kBlockM - 1) / kBlockM;
  if (ntiles > kBwdMaxTiles) return CPTHD_ERR_UNSUPPORTED;
  if (dk_dev == nullptr || dv_dev == nullptr || (T > 0 && k_dev == nullptr)) return CPTHD_ERR_INVALID_ARG;
  // every host check comes before the first thing queued on the stream: a
  // call that returns an error has touched nothing
  if (t_local > 0) {
    if (q_slice_idx_dev == nullptr || q_dev == nullptr || v_dev == nullptr || out_dev == nullptr ||
        dout_dev == nullptr || lse_dev == nullptr || cu_seqlens_dev == nullptr || dq_dev == nullptr ||
        num_docs < 1 || T < 1)
      return CPTHD_ERR_INVALID_ARG;
    const uintptr_t align = reinterpret_cast<uintptr_t>(q_dev) | reinterpret_cast<uintptr_t>(k_dev) |
                            reinterpret_cast<uintptr_t>(v_dev) | reinterpret_cast<uintptr_t>(dout_dev) |
                            reinterpret_cast<uintptr_t>(dq_dev) | reinterpret_cast<uintptr_t>(dk_dev) |
                            reinterpret_cast<uintptr_t>(dv_dev);
    if (align & 15) return CPTHD_ERR_UNSUPPORTED;
    if (workspace_dev == nullptr || workspace_bytes < bwd_workspace_bytes(ntiles, Hq) ||
        (reinterpret_cast<uintptr_t>(workspace_dev) & 255))
      return CPTHD_ERR_WORKSPACE;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // An empty slice contributes nothing: dK/dV are zero. Otherwise the dK/dV
  // pass writes every key tile, zeros where no query of the slice reaches.
  if (t_local == 0) {
    CPTHD_TRY_CUDA(cudaMemsetAsync(dk_dev, 0, sizeof(float) * static_cast<size_t>(T) * Hkv * d, s));
    CPTHD_TRY_CUDA(cudaMemsetAsync(dv_dev, 0, sizeof(float) * static_cast<size_t>(T) * Hkv * d, s));
    return CPTHD_OK;
  }
  const int32_t* cup = cu_seqlens_padded_dev ? cu_seqlens_padded_dev : cu_seqlens_dev;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf(static_cast<float>(d));
  AttnWorkspace ws = carve_workspace(workspace_dev, ntiles, kBlockM);
  char* extra = static_cast<char*>(workspace_dev) + attn_workspace_bytes(ntiles, kBlockM);
  float* lse2 = reinterpret_cast<float*>(extra);
  float* dvec = reinterpret_cast<float*>(extra + align256(sizeof(float) * ntiles * kBlockM * Hq));
  int32_t* work = reinterpret_cast<int32_t*>(extra + 2 * align256(sizeof(float) * ntiles * kBlockM * Hq));
  uint8_t* aug = reinterpret_cast<uint8_t*>(extra + 2 * align256(sizeof(float) * ntiles * kBlockM * Hq) +
                                            align256(sizeof(int32_t) * 8));
  attn_group_meta_kernel<kBlockM><<<static_cast<unsigned>(ntiles), kBlockM, 0, s>>>(
      index_list(q_slice_idx_dev), t_local, cu_seqlens_dev, cup, num_docs, T, ws, err_dev);
  CPTHD_TRY_CUDA(cudaGetLastError());
  if (d == 128)
    return launch_bwd<128>(q_dev, k_dev, v_dev, out_dev, dout_dev, lse_dev, t_local, T, Hq, Hkv, scale, ws, lse2,
                           dvec, aug, work, ntiles, dq_dev, dk_dev, dv_dev, err_dev, s);
  return launch_bwd<64>(q_dev, k_dev, v_dev, out_dev, dout_dev, lse_dev, t_local, T, Hq, Hkv, scale, ws, lse2, dvec,
                        aug, work, ntiles, dq_dev, dk_dev, dv_dev, err_dev, s);
}
