// 4-bit group quantiser and hybrid-cache construction.
//
// Quant_B(.; G) of Algorithm 4 ("HyQuant: Hybrid-Precision Quantization for
// LLM Attention", Appendix A.4) with B = 4 and G = 32 along head_dim, and the
// Freeze re-organisation of the cache into a 4-bit stream, vertical-line rows
// and a BF16 tail (§4.3 Eq. 8).
//
// A CTA builds one 64-row block of the 4-bit stream: the BF16 rows are staged
// in shared memory with each group's min / max, one thread per group derives
// the FP16 step and zero point, and each thread then assembles whole 32-bit
// code words in the tensor-core fragment order documented in hyq.h and
// stores them directly (no atomics, no float64).
#include "hyq_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRows = HYQ_QBLOCK_ROWS;  // 64 stream rows per block
constexpr int kChunks = HYQ_D / 8;      // 16 chunks of 8 elements per row

// Shared image of one 64-row block being built.
struct BuildSmem {
  __nv_bfloat16 x[2][kRows][HYQ_D];  // K and V rows (zero for padding / kept rows)
  float mn[2][kRows][4], mx[2][kRows][4];
  float s[2][kRows][4], z[2][kRows][4], r[2][kRows][4];
  int32_t pos[kRows];      // source row of each slot, -1 for none
  uint8_t keep[kRows];     // slot already holds a stream row (append)
  uint8_t nan[2][kRows][4];
};

__device__ __forceinline__ uint32_t code_of(float x, float s, float z, float r) {
  if (s == 0.f) return 0u;
  float t = rintf(__fmul_rn(__fsub_rn(x, z), r));
  t = fminf(fmaxf(t, 0.f), 15.f);
  return (uint32_t)t;
}

__device__ __forceinline__ void unpack8(uint4 v, float (&f)[8]) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(p[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// Build one 64-row block of the 4-bit stream at `dst` (10240 bytes, global).
// sm.pos / sm.keep must be set.  Rows with keep = 1 keep their existing
// codes and metadata; rows with pos < 0 become zero padding.
__device__ void build_block(BuildSmem& sm, const __nv_bfloat16* kbase, const __nv_bfloat16* vbase,
                            uint8_t* dst, bool any_keep, int32_t* err) {
  const int tid = threadIdx.x;
  // Pass 1: load the rows (all of a thread's loads first), per-group min /
  // max (4 chunks of 8 per group are on 4 consecutive lanes).
  constexpr int kPer = 2 * kRows * kChunks / kThreads;
  uint4 vin[kPer];
#pragma unroll
  for (int it = 0; it < kPer; ++it) {
    const int f = tid + it * kThreads;
    const int T = f >> 10, row = (f >> 4) & (kRows - 1), c = f & (kChunks - 1);
    const int32_t p = sm.pos[row];
    vin[it] = make_uint4(0, 0, 0, 0);
    if (p >= 0 && !sm.keep[row])
      vin[it] = __ldg(reinterpret_cast<const uint4*>((T ? vbase : kbase) + (size_t)p * HYQ_D + 8 * c));
  }
#pragma unroll
  for (int it = 0; it < kPer; ++it) {
    const int f = tid + it * kThreads;
    const int T = f >> 10, row = (f >> 4) & (kRows - 1), c = f & (kChunks - 1);
    const uint4 v = vin[it];
    *reinterpret_cast<uint4*>(&sm.x[T][row][8 * c]) = v;
    float e[8];
    unpack8(v, e);
    float mn = e[0], mx = e[0];
    int nan = isnan(e[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i) {
      mn = fminf(mn, e[i]);
      mx = fmaxf(mx, e[i]);
      nan |= isnan(e[i]);
    }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      nan |= __shfl_xor_sync(0xffffffffu, nan, o);
    }
    if ((c & 3) == 0) {
      sm.mn[T][row][c >> 2] = mn;
      sm.mx[T][row][c >> 2] = mx;
      sm.nan[T][row][c >> 2] = (uint8_t)nan;
    }
  }
  __syncthreads();
  // Pass 2: one thread per group: step s = smallest FP16 with 15 s >= mx - mn
  // (the subtraction, the division and the FP16 conversion all round up,
  // which gives exactly that value); zero z = FP16(mn) to nearest.
  for (int i = tid; i < 2 * kRows * 4; i += kThreads) {
    const int T = i >> 8, row = (i >> 2) & (kRows - 1), q = i & 3;
    if (sm.keep[row]) continue;
    const float mn = sm.mn[T][row][q], mx = sm.mx[T][row][q];
    __half sh = __float2half_ru(__fdiv_ru(__fsub_ru(mx, mn), 15.f));
    __half zh = __float2half_rn(mn);
    float s32 = __half2float(sh), z32 = __half2float(zh);
    if (sm.nan[T][row][q] || isinf(s32) || isinf(z32)) {
      hyq_set_err(err, HYQ_DEVERR_QUANT_RANGE);
      sh = zh = __float2half_rn(0.f);
      s32 = z32 = 0.f;
    }
    sm.s[T][row][q] = s32;
    sm.z[T][row][q] = z32;
    sm.r[T][row][q] = s32 > 0.f ? __frcp_rn(s32) : 0.f;
    const uint32_t w = (uint32_t)__half_as_ushort(sh) | ((uint32_t)__half_as_ushort(zh) << 16);
    *reinterpret_cast<uint32_t*>(dst + (row >> 4) * HYQ_QTILE_BYTES + 2048 + T * 256 + (row & 15) * 16 + 4 * q) = w;
  }
  __syncthreads();
  // Pass 3a: K code words.  Job (tile, g, chunk cc): rows g and g+8 of the
  // tile, elements 8cc..8cc+7 -> the two words u = 2(cc/4) + {0,1} of lane 4g + cc%4.
  for (int j = tid; j < 4 * 8 * kChunks; j += kThreads) {
    const int tile = j >> 7, g = (j >> 4) & 7, cc = j & 15;
    const int q = cc >> 2, t = cc & 3;
    uint8_t* wp = dst + tile * HYQ_QTILE_BYTES + 512 * (cc >> 3) + 16 * (4 * g + t) + 4 * (2 * (q & 1));
    uint32_t w[2] = {0u, 0u};
    uint2 old = make_uint2(0, 0);
    if (any_keep) old = *reinterpret_cast<const uint2*>(wp);
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const int row = 16 * tile + g + 8 * a;
      if (sm.keep[row]) {
        const uint32_t mm = 0x0F0F0F0Fu << (4 * a);  // this row's nibbles a + 2b + 4c
        w[0] |= old.x & mm;
        w[1] |= old.y & mm;
        continue;
      }
      float e[8];
      unpack8(*reinterpret_cast<const uint4*>(&sm.x[0][row][8 * cc]), e);
      const float s = sm.s[0][row][q], z = sm.z[0][row][q], r = sm.r[0][row][q];
#pragma unroll
      for (int sub = 0; sub < 2; ++sub)
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
          for (int c = 0; c < 2; ++c)
            w[sub] |= code_of(e[4 * sub + 2 * b + c], s, z, r) << (4 * (a + 2 * b + 4 * c));
    }
    *reinterpret_cast<uint2*>(wp) = make_uint2(w[0], w[1]);
  }
  // Pass 3b: V code words.  Job (tile, t, chunk cc): rows 2t + 8b + c,
  // elements 8cc..8cc+7 = 32q + 4g + 2s + a with q = cc/4 and g = 2(cc%4) + gl
  // -> the words (lane 4g + t, u = 2q + s) for gl, s in {0, 1}; the two s
  // words of one lane are adjacent.
  for (int j = tid; j < 4 * 4 * kChunks; j += kThreads) {
    const int tile = j >> 6, t = (j >> 4) & 3, cc = j & 15;
    const int q = cc >> 2;
    uint8_t* wp[2];
    uint32_t w[2][2] = {{0u, 0u}, {0u, 0u}};
    uint2 old[2] = {make_uint2(0, 0), make_uint2(0, 0)};
#pragma unroll
    for (int gl = 0; gl < 2; ++gl) {
      const int g = 2 * (cc & 3) + gl;
      wp[gl] = dst + tile * HYQ_QTILE_BYTES + 1024 + 512 * (cc >> 3) + 16 * (4 * g + t) + 8 * (q & 1);
      if (any_keep) old[gl] = *reinterpret_cast<const uint2*>(wp[gl]);
    }
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int row = 16 * tile + 2 * t + 8 * b + c;
        if (sm.keep[row]) {
          const uint32_t mm = 0xFFu << (4 * (2 * b + 4 * c));  // nibbles a + 2b + 4c, a = 0, 1
#pragma unroll
          for (int gl = 0; gl < 2; ++gl) {
            w[gl][0] |= old[gl].x & mm;
            w[gl][1] |= old[gl].y & mm;
          }
          continue;
        }
        float e[8];
        unpack8(*reinterpret_cast<const uint4*>(&sm.x[1][row][8 * cc]), e);
        const float s = sm.s[1][row][q], z = sm.z[1][row][q], r = sm.r[1][row][q];
#pragma unroll
        for (int gl = 0; gl < 2; ++gl)
#pragma unroll
          for (int ss = 0; ss < 2; ++ss)
#pragma unroll
            for (int a = 0; a < 2; ++a)
              w[gl][ss] |= code_of(e[4 * gl + 2 * ss + a], s, z, r) << (4 * (a + 2 * b + 4 * c));
      }
#pragma unroll
    for (int gl = 0; gl < 2; ++gl) *reinterpret_cast<uint2*>(wp[gl]) = make_uint2(w[gl][0], w[gl][1]);
  }
}

// Source position of stream row r: the r-th position of [0, P) not in idx
// (idx strictly ascending).  With f(i) = idx[i] - i non-decreasing, the
// number of idx entries before that position is #{i : f(i) <= r}.
__device__ __forceinline__ int32_t stream_pos(int32_t r, const int32_t* idx, int32_t k) {
  int32_t lo = 0, hi = k;
  while (lo < hi) {
    int32_t mid = (lo + hi) >> 1;
    if (idx[mid] - mid <= r) lo = mid + 1;
    else hi = mid;
  }
  return r + lo;
}

// Warp-cooperative #{i < k : idx[i] - i <= x} for a strictly ascending idx
// (so idx[i] - i is non-decreasing): 32 probes per round.
__device__ __forceinline__ int32_t warp_count_f_le(const int32_t* idx, int32_t k, int32_t x, int lane) {
  int32_t lo = 0, hi = k;  // f(i) <= x for i < lo, f(i) > x for i >= hi
  while (lo < hi) {
    const int32_t step = (hi - lo + 31) >> 5;
    const int32_t i = lo + lane * step;
    const bool le = i < hi && __ldg(idx + i) - i <= x;
    const int cnt = __popc(__ballot_sync(0xffffffffu, le));
    if (cnt == 0) {
      hi = lo;
    } else {
      const int32_t nlo = lo + (cnt - 1) * step + 1;
      hi = min(hi, lo + cnt * step);
      lo = nlo;
    }
  }
  return lo;
}

constexpr int kWinF = 256;  // vertical-line entries a block resolves in shared memory

// grid (blocks of the new stream, HKV, B)
__global__ void __launch_bounds__(kThreads) rebuild_blocks_kernel(
    const __nv_bfloat16* __restrict__ k_src, const __nv_bfloat16* __restrict__ v_src, int32_t ld,
    int32_t P, const int32_t* __restrict__ idx, int32_t k, uint8_t* __restrict__ qblocks,
    int32_t nblk_cap, int32_t* err) {
  __shared__ __align__(16) BuildSmem sm;
  const int bi = blockIdx.x, h = blockIdx.y, b = blockIdx.z, HKV = gridDim.y;
  const size_t bh = (size_t)b * HKV + h;
  const int32_t nq = P - k;
  const int32_t* idx_bh = idx ? idx + bh * k : nullptr;
  // Stream row R sits at position R + #{i : idx[i] - i <= R}.  Warps 0 and 1
  // find that count at the block's first and last row; the entries in
  // between go to shared memory, where every row counts its own.
  __shared__ int32_t s_c[2];
  __shared__ int32_t s_f[kWinF];
  const int32_t r0 = bi * kRows, r1 = min(nq, r0 + kRows) - 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (k > 0 && warp < 2) {
    const int32_t c = warp_count_f_le(idx_bh, k, warp == 0 ? r0 - 1 : r1, lane);
    if (lane == 0) s_c[warp] = c;
  }
  __syncthreads();
  const int32_t c0 = k > 0 ? s_c[0] : 0, m = k > 0 ? s_c[1] - s_c[0] : 0;
  if (m <= kWinF)
    for (int i = threadIdx.x; i < m; i += kThreads) s_f[i] = __ldg(idx_bh + c0 + i) - (c0 + i);
  __syncthreads();
  if (threadIdx.x < kRows) {
    const int32_t r = bi * kRows + threadIdx.x;
    int32_t p = -1;
    if (r < nq) {
      if (k == 0) {
        p = r;
      } else if (m <= kWinF) {
        int32_t c = c0;
        for (int i = 0; i < m; ++i) c += s_f[i] <= r;
        p = r + c;
      } else {
        p = stream_pos(r, idx_bh, k);  // a run of more than kWinF vertical lines
      }
      if (p < 0 || p >= P) {  // only possible for an invalid idx list
        hyq_set_err(err, HYQ_DEVERR_INDEX);
        p = min(max(p, 0), P - 1);
      }
    }
    sm.pos[threadIdx.x] = p;
    sm.keep[threadIdx.x] = 0;
  }
  __syncthreads();
  build_block(sm, k_src + bh * ld * HYQ_D, v_src + bh * ld * HYQ_D,
              qblocks + (bh * nblk_cap + bi) * (size_t)HYQ_QBLOCK_BYTES, false, err);
}

// Vertical-line gather, BF16 tail copy and counters.  One warp per row:
// lanes 0-15 copy the K row, lanes 16-31 the V row.  grid (ceil((k+ntail)/8), HKV, B)
__global__ void __launch_bounds__(kThreads) rebuild_gather_kernel(
    const __nv_bfloat16* __restrict__ k_src, const __nv_bfloat16* __restrict__ v_src, int32_t ld,
    int32_t L, int32_t P, const int32_t* __restrict__ idx, int32_t k, hyq_layout lay,
    int32_t cap_vl, int32_t cap_tail) {
  const int h = blockIdx.y, b = blockIdx.z, HKV = gridDim.y;
  const size_t bh = (size_t)b * HKV + h;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t ntail = L - P;
  const int32_t row = blockIdx.x * kWarps + warp;
  if (row < k + ntail) {
    int32_t src;
    uint4* dk;
    uint4* dv;
    if (row < k) {
      src = idx[bh * k + row];
      bool ok = src >= 0 && src < P && (row == 0 || idx[bh * k + row - 1] < src);
      if (!ok) {
        if (lane == 0) hyq_set_err(lay.err, HYQ_DEVERR_INDEX);
        src = min(max(src, 0), max(P - 1, 0));
      }
      dk = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(lay.vl_k) + (bh * cap_vl + row) * HYQ_D);
      dv = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(lay.vl_v) + (bh * cap_vl + row) * HYQ_D);
      if (lane == 0) lay.vl_idx[bh * cap_vl + row] = src;
    } else {
      int32_t t = row - k;
      src = P + t;
      dk = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(lay.tail_k) + (bh * cap_tail + t) * HYQ_D);
      dv = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(lay.tail_v) + (bh * cap_tail + t) * HYQ_D);
    }
    const uint4* s = reinterpret_cast<const uint4*>((lane < 16 ? k_src : v_src) + (bh * ld + src) * HYQ_D);
    (lane < 16 ? dk : dv)[lane & 15] = s[lane & 15];
  }
  if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0) {
    int32_t* cnt = lay.counts + (size_t)b * HYQ_COUNTS;
    cnt[HYQ_CNT_NQ] = P - k;
    cnt[HYQ_CNT_NVL] = k;
    cnt[HYQ_CNT_NTAIL] = ntail;
    cnt[HYQ_CNT_LEN] = L;
  }
}

// Append n rows per (b, h) after the current NQ rows.  grid (blocks touched, HKV, B)
__global__ void __launch_bounds__(kThreads) append_blocks_kernel(
    const __nv_bfloat16* __restrict__ k_rows, const __nv_bfloat16* __restrict__ v_rows, int32_t n,
    hyq_layout lay, int32_t nblk_cap) {
  __shared__ __align__(16) BuildSmem sm;
  const int h = blockIdx.y, b = blockIdx.z, HKV = gridDim.y;
  const size_t bh = (size_t)b * HKV + h;
  const int32_t nq0 = lay.counts[(size_t)b * HYQ_COUNTS + HYQ_CNT_NQ];
  const int32_t cap_rows = nblk_cap * kRows;
  if (nq0 < 0 || nq0 > cap_rows) {
    if (threadIdx.x == 0) hyq_set_err(lay.err, HYQ_DEVERR_COUNT);
    return;
  }
  const int32_t end = min(nq0 + n, cap_rows);
  if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0 && nq0 + n > cap_rows)
    hyq_set_err(lay.err, HYQ_DEVERR_COUNT);
  const int32_t bi = nq0 / kRows + blockIdx.x;
  if (max(bi * kRows, nq0) >= min((bi + 1) * kRows, end)) return;  // uniform across the block
  if (threadIdx.x < kRows) {
    const int32_t row = bi * kRows + threadIdx.x;
    sm.keep[threadIdx.x] = row < nq0;
    sm.pos[threadIdx.x] = (row >= nq0 && row < end) ? row - nq0 : -1;
  }
  __syncthreads();
  build_block(sm, k_rows + bh * n * HYQ_D, v_rows + bh * n * HYQ_D,
              lay.qblocks + (bh * nblk_cap + bi) * (size_t)HYQ_QBLOCK_BYTES, bi * kRows < nq0, lay.err);
}

__global__ void append_counts_kernel(hyq_layout lay, int32_t n, int32_t cap_rows) {
  const int b = blockIdx.x;
  int32_t* cnt = lay.counts + (size_t)b * HYQ_COUNTS;
  int32_t nq0 = cnt[HYQ_CNT_NQ];
  if (nq0 < 0 || nq0 > cap_rows) return;
  int32_t add = min(n, cap_rows - nq0);
  cnt[HYQ_CNT_NQ] = nq0 + add;
  cnt[HYQ_CNT_LEN] += add;
}

}  // namespace

cudaError_t hyq_launch_quantize_append(const hyq_config* c, const void* k, const void* v,
                                       int32_t n_rows, const hyq_layout* lay, cudaStream_t s) {
  int32_t nblk = hyq_nblk(c);
  dim3 grid((n_rows + HYQ_QBLOCK_ROWS - 1) / HYQ_QBLOCK_ROWS + 1, c->num_kv_heads, c->batch);
  append_blocks_kernel<<<grid, kThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(k),
                                                 static_cast<const __nv_bfloat16*>(v), n_rows,
                                                 *lay, nblk);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  append_counts_kernel<<<c->batch, 1, 0, s>>>(*lay, n_rows, nblk * HYQ_QBLOCK_ROWS);
  return cudaGetLastError();
}

cudaError_t hyq_launch_rebuild(const hyq_config* c, const void* k_src, const void* v_src,
                               int32_t ld, int32_t L, const int32_t* idx, int32_t k,
                               const hyq_layout* lay, cudaStream_t s) {
  int32_t P = L - c->window > 0 ? L - c->window : 0;
  int32_t nq = P - k;
  int32_t nblk = hyq_nblk(c);
  const __nv_bfloat16* kk = static_cast<const __nv_bfloat16*>(k_src);
  const __nv_bfloat16* vv = static_cast<const __nv_bfloat16*>(v_src);
  if (nq > 0) {
    dim3 grid((nq + HYQ_QBLOCK_ROWS - 1) / HYQ_QBLOCK_ROWS, c->num_kv_heads, c->batch);
    rebuild_blocks_kernel<<<grid, kThreads, 0, s>>>(kk, vv, ld, P, idx, k, lay->qblocks, nblk, lay->err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  int32_t rows = k + (L - P);
  dim3 grid2(rows > 0 ? (rows + kWarps - 1) / kWarps : 1, c->num_kv_heads, c->batch);
  rebuild_gather_kernel<<<grid2, kThreads, 0, s>>>(kk, vv, ld, L, P, idx, k, *lay, hyq_vl_stride(c),
                                                   hyq_cap_tail(c));
  return cudaGetLastError();
}
