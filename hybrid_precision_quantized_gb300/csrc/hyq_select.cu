// Vertical-line token identification ("HyQuant: Hybrid-Precision
// Quantization for LLM Attention", §4.1 Eq. 4-5 and Appendix A.1
// Algorithm 1), per KV head:
//   u    = sum of the proxy queries of the g query heads of the group
//   S(j) = u . k_j for j < P = max(0, L - W)             (float32)
//   idx  = the k positions of largest S, ties to the lower position,
//          written in ascending order.
// Three launches: proxy sum, scores (HBM-bound pass over the BF16 keys),
// radix select + ordered compaction (one CTA per KV head).
#include "hyq_common.cuh"

namespace {

constexpr int kScoreThreads = 256;
constexpr int kScoreRowsPerCta = 64;
constexpr int kTopkThreads = 1024;

struct SelectWs {
  int32_t* err;
  float* u;        // [B][HKV][128]
  uint32_t* keys;  // [B][HKV][Pmax]
};

size_t round_up(size_t x) { return (x + 255) / 256 * 256; }

SelectWs carve(const hyq_config* c, int32_t L, void* ws) {
  size_t bh = (size_t)c->batch * c->num_kv_heads;
  char* p = static_cast<char*>(ws);
  SelectWs w;
  w.err = reinterpret_cast<int32_t*>(p);
  p += 256;
  w.u = reinterpret_cast<float*>(p);
  p += round_up(bh * HYQ_D * 4);
  w.keys = reinterpret_cast<uint32_t*>(p);
  (void)L;
  return w;
}

// u[b][kvh][d] = sum over t < n_proxy and the g heads of the group.  grid (HKV, B), 128 threads
__global__ void proxy_sum_kernel(const __nv_bfloat16* __restrict__ qp, int32_t n_proxy,
                                 int32_t n_ld, int32_t gq, float* __restrict__ u) {
  const int h = blockIdx.x, b = blockIdx.y, HKV = gridDim.x, d = threadIdx.x;
  float acc = 0.f;
  for (int j = 0; j < gq; ++j) {
    const __nv_bfloat16* base = qp + (((size_t)b * HKV * gq + (size_t)h * gq + j) * n_ld) * HYQ_D + d;
    for (int t = 0; t < n_proxy; ++t) acc += __bfloat162float(base[(size_t)t * HYQ_D]);
  }
  u[((size_t)b * HKV + h) * HYQ_D + d] = acc;
}

__device__ __forceinline__ uint32_t order_key(float s, int32_t* err) {
  if (isnan(s)) {
    hyq_set_err(err, HYQ_DEVERR_SCORE);
    return 0u;
  }
  if (s == 0.f) s = 0.f;  // -0 and +0 compare equal
  uint32_t bits = __float_as_uint(s);
  return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
}

// One half-warp per key row (16 lanes x 8 elements).  grid (ceil(P/64), HKV, B)
__global__ void __launch_bounds__(kScoreThreads) score_kernel(
    const __nv_bfloat16* __restrict__ k_src, int32_t ld, int32_t P, const float* __restrict__ u,
    uint32_t* __restrict__ keys, int32_t pmax, int32_t* err) {
  const int h = blockIdx.y, b = blockIdx.z, HKV = gridDim.y;
  const size_t bh = (size_t)b * HKV + h;
  const int lane = threadIdx.x & 31, half = lane >> 4, sub = lane & 15;
  const int warp = threadIdx.x >> 5;
  float uu[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) uu[i] = u[bh * HYQ_D + 8 * sub + i];
  const __nv_bfloat16* kb = k_src + bh * ld * HYQ_D;
  const int end = min(P, (int)(blockIdx.x + 1) * kScoreRowsPerCta);
  // The trip count is uniform across the warp (both half-warps run every
  // iteration) so the full-mask shuffles below are always complete.
  for (int r0 = blockIdx.x * kScoreRowsPerCta + 2 * warp; r0 < end; r0 += 2 * (kScoreThreads / 32)) {
    const int r = r0 + half;
    const bool valid = r < end;
    float s = 0.f;
    if (valid) {
      uint4 raw = *reinterpret_cast<const uint4*>(kb + (size_t)r * HYQ_D + 8 * sub);
      const __nv_bfloat162* pr = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(pr[i]);
        s = fmaf(uu[2 * i], f.x, s);
        s = fmaf(uu[2 * i + 1], f.y, s);
      }
    }
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (valid && sub == 0) keys[bh * pmax + r] = order_key(s, err);
  }
}

// Block-wide exclusive scan of 0/1 flags (1024 threads).  Returns the prefix
// for this thread; *total gets the block total.
__device__ __forceinline__ int block_scan_flag(int f, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned m = __ballot_sync(0xffffffffu, f);
  int pre = __popc(m & ((1u << lane) - 1u));
  if (lane == 0) warp_sums[warp] = __popc(m);
  __syncthreads();
  if (warp == 0) {
    int v = warp_sums[lane];
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    warp_sums[lane] = x - v;  // exclusive
    if (lane == 31) warp_sums[32] = x;
  }
  __syncthreads();
  int r = warp_sums[warp] + pre;
  *total = warp_sums[32];
  __syncthreads();
  return r;
}

// Radix select of the k-th largest key, then the ordered compaction of the
// selected positions.  grid (HKV, B), 1024 threads.
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const uint32_t* __restrict__ keys,
                                                            int32_t pmax, int32_t P, int32_t k,
                                                            int32_t* __restrict__ idx_out) {
  __shared__ int hist[256];
  __shared__ int warp_sums[33];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining;
  const int h = blockIdx.x, b = blockIdx.y, HKV = gridDim.x;
  const size_t bh = (size_t)b * HKV + h;
  const uint32_t* kk = keys + bh * pmax;
  uint32_t prefix = 0, mask = 0;
  int remaining = k;  // how many still to take among keys matching the prefix
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < P; j += kTopkThreads) {
      uint32_t key = kk[j];
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // Find the digit D (from the top) where the running count reaches `remaining`.
      int lane = threadIdx.x;
      int above = 0, digit = -1, rem = remaining;
      for (int base = 255; base >= 0 && digit < 0; base -= 32) {
        int bin = base - lane;
        int c = hist[bin];
        int x = c;  // inclusive scan from the top down the 32 bins
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          int y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        unsigned hit = __ballot_sync(0xffffffffu, above + x >= rem);
        if (hit) {
          int first = __ffs(hit) - 1;
          int excl = __shfl_sync(0xffffffffu, x - c, first);
          digit = base - first;
          rem -= above + excl;
        } else {
          above += __shfl_sync(0xffffffffu, x, 31);
        }
      }
      if (lane == 0) {
        s_prefix = prefix | ((uint32_t)digit << shift);
        s_remaining = rem;
      }
    }
    __syncthreads();
    prefix = s_prefix;
    remaining = s_remaining;
    mask |= 255u << shift;
    __syncthreads();
  }
  // prefix = threshold key T; take every key > T and the first `remaining`
  // keys equal to T in position order.
  const uint32_t T = prefix;
  int eq_base = 0, out_base = 0, total;
  int32_t* out = idx_out + bh * k;
  for (int j0 = 0; j0 < P; j0 += kTopkThreads) {
    int j = j0 + threadIdx.x;
    uint32_t key = j < P ? kk[j] : 0u;
    int eq = (j < P) && key == T;
    int eq_rank = block_scan_flag(eq, warp_sums, &total);
    int take = (j < P) && (key > T || (eq && eq_base + eq_rank < remaining));
    eq_base += total;
    int pos = block_scan_flag(take, warp_sums, &total);
    if (take && out_base + pos < k) out[out_base + pos] = j;
    out_base += total;
  }
}

}  // namespace

size_t hyq_select_ws_bytes(const hyq_config* c, int32_t L) {
  size_t bh = (size_t)c->batch * c->num_kv_heads;
  int32_t P = L - c->window > 0 ? L - c->window : 0;
  return 256 + round_up(bh * HYQ_D * 4) + round_up(bh * (size_t)(P > 0 ? P : 1) * 4);
}

cudaError_t hyq_launch_select(const hyq_config* c, const void* q_proxy, int32_t n_proxy,
                              int32_t n_proxy_ld, const void* k_src, int32_t ld, int32_t L,
                              int32_t* idx_out, int32_t k, void* ws, cudaStream_t s) {
  SelectWs w = carve(c, L, ws);
  const int32_t P = L - c->window;  // > 0 since k > 0
  const int32_t gq = c->num_q_heads / c->num_kv_heads;
  proxy_sum_kernel<<<dim3(c->num_kv_heads, c->batch), HYQ_D, 0, s>>>(
      static_cast<const __nv_bfloat16*>(q_proxy), n_proxy, n_proxy_ld, gq, w.u);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 g2((P + kScoreRowsPerCta - 1) / kScoreRowsPerCta, c->num_kv_heads, c->batch);
  score_kernel<<<g2, kScoreThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(k_src), ld, P, w.u,
                                            w.keys, P, w.err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  topk_kernel<<<dim3(c->num_kv_heads, c->batch), kTopkThreads, 0, s>>>(w.keys, P, P, k, idx_out);
  return cudaGetLastError();
}
