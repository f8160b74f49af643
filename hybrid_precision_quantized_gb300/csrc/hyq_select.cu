// Vertical-line token identification ("HyQuant: Hybrid-Precision
// Quantization for LLM Attention", §4.1 Eq. 4-5 and Appendix A.1
// Algorithm 1), per KV head:
//   u    = sum of the proxy queries of the g query heads of the group
//   S(j) = u . k_j for j < P = max(0, L - W)             (float32)
//   idx  = the k positions of largest S, ties to the lower position,
//          written in ascending order.
// Three launches: proxy sum, scores (HBM-bound pass over the BF16 keys),
// radix select + ordered compaction (one CTA per KV head).
//
// Per query head (hyq_config.vl_mode = 1, Algorithm 1's B x H_Q x k sets):
// the proxies are summed per query head as well, one pass over the keys
// scores every query head of the group and the group itself, a top-k per
// query head gives the heads' sets, their positions are raised to the top
// key value in the group's scores, and a top-ku of those gives the stored
// per-KV-head list: the union of the group's sets, filled up to
// ku = min(P, g k) by the group score.
#include <cooperative_groups.h>

#include <algorithm>
#include <cmath>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "hyq_common.cuh"
#include "hyq_f2.cuh"
#include "hyq_tc.cuh"

namespace {

constexpr int kScoreThreads = 256;
constexpr int kScoreRowsPerCta = 64;
constexpr int kScoreRowsPerStep = 2 * (kScoreThreads / 32);  // one row per half-warp
constexpr int kScoreSteps = kScoreRowsPerCta / kScoreRowsPerStep;
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

// u[b][kvh][d] = sum over t < n_proxy and the g heads of the group.
// grid (HKV, B), 512 threads: thread (r, c) sums 8 dims (c) over the rows
// r, r + 32, ... of the g * n_proxy query rows with 16-byte loads; the 32
// row-group partials are then added in a fixed order (deterministic).
constexpr int kProxyThreads = 512;
__global__ void __launch_bounds__(kProxyThreads) proxy_sum_kernel(const __nv_bfloat16* __restrict__ qp,
                                                                  int32_t n_proxy, int32_t n_ld, int32_t gq,
                                                                  float* __restrict__ u) {
  __shared__ float part[32][HYQ_D + 4];
  const int h = blockIdx.x, b = blockIdx.y, HKV = gridDim.x;
  const int r0 = threadIdx.x >> 4, c = threadIdx.x & 15;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  const int rows = gq * n_proxy;
  // rows r0, r0 + 32, ... in order; eight of them loaded at a time
  for (int rb = r0; rb < rows; rb += 8 * 32) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int r = rb + 32 * u;
      v[u] = make_uint4(0, 0, 0, 0);
      if (r < rows) {
        const int j = r / n_proxy, t = r - j * n_proxy;
        const __nv_bfloat16* row = qp + (((size_t)b * HKV * gq + (size_t)h * gq + j) * n_ld + t) * HYQ_D;
        v[u] = __ldg(reinterpret_cast<const uint4*>(row) + c);
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (rb + 32 * u >= rows) break;
      const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&v[u]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(p2[i]);
        acc[2 * i] += f.x;
        acc[2 * i + 1] += f.y;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) part[r0][8 * c + i] = acc[i];
  __syncthreads();
  if (threadIdx.x < HYQ_D) {
    float s = 0.f;
    for (int r = 0; r < 32; ++r) s += part[r][threadIdx.x];
    u[((size_t)b * HKV + h) * HYQ_D + threadIdx.x] = s;
  }
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
  // A thread's rows (every 16th of the block's) are all loaded before the
  // first is reduced, so that they are in flight together.  Every lane runs
  // every step, so the full-mask shuffles below are always complete.
  uint4 raw[kScoreSteps];
#pragma unroll
  for (int it = 0; it < kScoreSteps; ++it) {
    const int r = blockIdx.x * kScoreRowsPerCta + it * kScoreRowsPerStep + 2 * warp + half;
    raw[it] = r < end ? *reinterpret_cast<const uint4*>(kb + (size_t)r * HYQ_D + 8 * sub) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int it = 0; it < kScoreSteps; ++it) {
    const int r = blockIdx.x * kScoreRowsPerCta + it * kScoreRowsPerStep + 2 * warp + half;
    const bool valid = r < end;
    float s = 0.f;
    if (valid) {
      const __nv_bfloat162* pr = reinterpret_cast<const __nv_bfloat162*>(&raw[it]);
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

// Scores of the g query heads of a KV head and of the group, one half-warp
// per key row as in score_kernel (the same operation order, so the group
// keys equal score_kernel's).  grid (ceil(P/64), HKV, B).
template <int G>
__global__ void __launch_bounds__(kScoreThreads) score_heads_kernel(
    const __nv_bfloat16* __restrict__ k_src, int32_t ld, int32_t P, const float* __restrict__ u_heads,
    const float* __restrict__ u_group, uint32_t* __restrict__ keys_heads, uint32_t* __restrict__ keys_group,
    int32_t* err) {
  const int h = blockIdx.y, b = blockIdx.z, HKV = gridDim.y;
  const size_t bh = (size_t)b * HKV + h;
  const int lane = threadIdx.x & 31, half = lane >> 4, sub = lane & 15;
  const int warp = threadIdx.x >> 5;
  float uu[G + 1][8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
#pragma unroll
    for (int r = 0; r < G; ++r) uu[r][i] = u_heads[(bh * G + r) * HYQ_D + 8 * sub + i];
    uu[G][i] = u_group[bh * HYQ_D + 8 * sub + i];
  }
  const __nv_bfloat16* kb = k_src + bh * ld * HYQ_D;
  const int end = min(P, (int)(blockIdx.x + 1) * kScoreRowsPerCta);
  uint4 raw[kScoreSteps];  // loaded together, as in score_kernel
#pragma unroll
  for (int it = 0; it < kScoreSteps; ++it) {
    const int r = blockIdx.x * kScoreRowsPerCta + it * kScoreRowsPerStep + 2 * warp + half;
    raw[it] = r < end ? *reinterpret_cast<const uint4*>(kb + (size_t)r * HYQ_D + 8 * sub) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int it = 0; it < kScoreSteps; ++it) {
    const int r = blockIdx.x * kScoreRowsPerCta + it * kScoreRowsPerStep + 2 * warp + half;
    const bool valid = r < end;
    float s[G + 1];
#pragma unroll
    for (int q = 0; q <= G; ++q) s[q] = 0.f;
    if (valid) {
      const __nv_bfloat162* pr = reinterpret_cast<const __nv_bfloat162*>(&raw[it]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(pr[i]);
#pragma unroll
        for (int q = 0; q <= G; ++q) {
          s[q] = fmaf(uu[q][2 * i], f.x, s[q]);
          s[q] = fmaf(uu[q][2 * i + 1], f.y, s[q]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q <= G; ++q)
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) s[q] += __shfl_xor_sync(0xffffffffu, s[q], o);
    if (valid && sub == 0) {
#pragma unroll
      for (int q = 0; q < G; ++q) keys_heads[(bh * G + q) * P + r] = order_key(s[q], err);
      keys_group[bh * P + r] = order_key(s[G], err);
    }
  }
}

// Raise the group keys of every position in a query head's set above any
// score key, so that a top-ku of the group keys takes the union first.
// grid (HQ, B).
__global__ void mark_union_kernel(const int32_t* __restrict__ idx_heads, int32_t k1, int32_t g, int32_t P,
                                  uint32_t* __restrict__ keys_group) {
  const int h = blockIdx.x, b = blockIdx.y, HQ = gridDim.x;
  const int32_t* ih = idx_heads + ((size_t)b * HQ + h) * k1;
  uint32_t* kg = keys_group + ((size_t)b * (HQ / g) + h / g) * P;
  for (int i = threadIdx.x; i < k1; i += blockDim.x) {
    const int32_t j = ih[i];
    if (j >= 0 && j < P) kg[j] = 0xFFFFFFFFu;  // above order_key(+inf)
  }
}

// Block-wide exclusive scan of small counts (1024 threads).  Returns the
// prefix for this thread; *total gets the block total.
__device__ __forceinline__ int block_scan_count(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int w = warp_sums[lane];
    int z = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, z, o);
      if (lane >= o) z += y;
    }
    warp_sums[lane] = z - w;
    if (lane == 31) warp_sums[32] = z;
  }
  __syncthreads();
  const int r = warp_sums[warp] + x - v;
  *total = warp_sums[32];
  __syncthreads();
  return r;
}

// Keys staged in shared memory when they fit (up to 200 KB).
constexpr int kTopkSmemKeys = 51200;

// Radix select of the k-th largest key, then the ordered compaction of the
// selected positions.  grid (HKV, B), 1024 threads.  The keys are read once
// into shared memory (when they fit); histogram updates are aggregated per
// warp (the high bytes of similar scores fall into few bins); the
// compaction takes 4 consecutive positions per thread per round.
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const uint32_t* __restrict__ keys,
                                                            int32_t pmax, int32_t P, int32_t k,
                                                            int32_t* __restrict__ idx_out) {
  extern __shared__ uint32_t skeys[];
  __shared__ int hist[256];
  __shared__ int warp_sums[33];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining;
  const int h = blockIdx.x, b = blockIdx.y, HKV = gridDim.x;
  const int lane = threadIdx.x & 31;
  const size_t bh = (size_t)b * HKV + h;
  const uint32_t* gk = keys + bh * pmax;
  const bool staged = P <= kTopkSmemKeys;
  if (staged) {
    for (int i = threadIdx.x; i < P; i += kTopkThreads) skeys[i] = gk[i];
    __syncthreads();
  }
  const uint32_t* kk = staged ? skeys : gk;
  uint32_t prefix = 0, mask = 0;
  int remaining = k;  // how many still to take among keys matching the prefix
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int j0 = 0; j0 < P; j0 += kTopkThreads) {  // uniform trip count for the warp vote
      const int j = j0 + threadIdx.x;
      const uint32_t key = j < P ? kk[j] : 0u;
      const bool in = j < P && (key & mask) == prefix;
      const int bin = in ? (int)((key >> shift) & 255u) : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, bin);
      if (in && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // Find the digit D (from the top) where the running count reaches `remaining`.
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
  for (int j0 = 0; j0 < P; j0 += 4 * kTopkThreads) {
    const int jb = j0 + 4 * threadIdx.x;
    uint32_t kv[4];
    bool eqf[4];
    int neq = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = jb + e;
      kv[e] = j < P ? kk[j] : 0u;
      eqf[e] = j < P && kv[e] == T;
      neq += eqf[e];
    }
    int eqr = eq_base + block_scan_count(neq, warp_sums, &total);
    eq_base += total;
    bool tk[4];
    int ntake = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      tk[e] = jb + e < P && (kv[e] > T || (eqf[e] && eqr < remaining));
      eqr += eqf[e];
      ntake += tk[e];
    }
    int o = out_base + block_scan_count(ntake, warp_sums, &total);
    out_base += total;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (tk[e]) {
        if (o < k) out[o] = jb + e;
        ++o;
      }
  }
}

// Cluster top-k: kTopkCluster blocks share one (sequence, KV head).  Block r
// holds positions [r * kTopkCtaThreads * KPT, ...) in registers, KPT
// consecutive positions per thread.  Each radix pass builds a local
// histogram; after a cluster barrier every block sums the kTopkCluster
// histograms over distributed shared memory and finds the same digit.  The
// selected positions are then written in position order: a key at global
// order j goes to out[#{greater before j} + min(#{equal before j}, remaining)],
// both counts from one packed block scan plus the counts of lower-ranked
// blocks.
constexpr int kTopkCluster = 8;
constexpr int kTopkCtaThreads = 512;
constexpr int kTopkCtaWarps = kTopkCtaThreads / 32;

template <int KPT>
__global__ void __cluster_dims__(kTopkCluster, 1, 1) __launch_bounds__(kTopkCtaThreads)
    topk_cluster_kernel(const uint32_t* __restrict__ keys, int32_t pmax, int32_t P, int32_t k,
                        int32_t* __restrict__ idx_out) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  __shared__ int hist[4][256];
  __shared__ int wsum[kTopkCtaWarps];
  __shared__ int s_cnt[2];  // this block's (greater, equal) counts
  __shared__ int s_base[2];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = (int)cl.block_rank();
  const size_t bh = (size_t)blockIdx.z * gridDim.y + blockIdx.y;
  const uint32_t* gk = keys + bh * pmax;
  const int32_t j0 = (rank * kTopkCtaThreads + tid) * KPT;
  uint32_t kv[KPT];
#pragma unroll
  for (int e = 0; e < KPT; ++e) kv[e] = j0 + e < P ? __ldg(gk + j0 + e) : 0u;
  for (int i = tid; i < 4 * 256; i += kTopkCtaThreads) (&hist[0][0])[i] = 0;
  __syncthreads();
  uint32_t prefix = 0, mask = 0;
  int remaining = k;  // 1 <= remaining <= #keys matching prefix
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
      const bool in = j0 + e < P && (kv[e] & mask) == prefix;
      if (__any_sync(0xffffffffu, in)) {
        const int bin = in ? (int)((kv[e] >> shift) & 255u) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, bin);
        if (in && lane == __ffs(peers) - 1) atomicAdd(&hist[pass][bin], __popc(peers));
      }
    }
    cl.sync();  // every block's histogram of this pass is complete
    int tot = 0, x = 0;
    if (tid < 256) {
#pragma unroll
      for (int c = 0; c < kTopkCluster; ++c) tot += cl.map_shared_rank(&hist[pass][0], c)[tid];
      x = tot;  // suffix sum over this warp's bins >= tid
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, x, o);
        if (lane + o < 32) x += y;
      }
      if (lane == 0) wsum[warp] = x;
    }
    __syncthreads();
    if (tid < 256) {
      int S = x;  // #keys matching prefix with digit >= tid
      for (int w = warp + 1; w < 8; ++w) S += wsum[w];
      if (S >= remaining && S - tot < remaining) {
        s_prefix = prefix | ((uint32_t)tid << shift);
        s_remaining = remaining - (S - tot);
      }
    }
    __syncthreads();
    prefix = s_prefix;
    remaining = s_remaining;
    mask |= 255u << shift;
  }
  const uint32_t T = prefix;
  int ngt = 0, neq = 0;
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    const bool valid = j0 + e < P;
    ngt += valid && kv[e] > T;
    neq += valid && kv[e] == T;
  }
  // Packed exclusive scan of (greater << 16 | equal); a block holds at most
  // kTopkCtaThreads * KPT <= 8192 keys, so neither half overflows.
  const int v = (ngt << 16) | neq;
  int xs = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, xs, o);
    if (lane >= o) xs += y;
  }
  __shared__ int wscan[kTopkCtaWarps];
  if (lane == 31) wscan[warp] = xs;
  __syncthreads();
  int excl = xs - v;
  for (int w = 0; w < warp; ++w) excl += wscan[w];
  if (tid == 0) {
    int t = 0;
    for (int w = 0; w < kTopkCtaWarps; ++w) t += wscan[w];
    s_cnt[0] = t >> 16;
    s_cnt[1] = t & 0xffff;
  }
  cl.sync();  // every block's counts are published
  if (warp == 0) {
    int g = 0, q = 0;
    if (lane < rank) {
      const int* rc = cl.map_shared_rank(s_cnt, lane);
      g = rc[0];
      q = rc[1];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      g += __shfl_xor_sync(0xffffffffu, g, o);
      q += __shfl_xor_sync(0xffffffffu, q, o);
    }
    if (lane == 0) {
      s_base[0] = g;
      s_base[1] = q;
    }
  }
  cl.barrier_arrive();  // this block reads no other block's shared memory after here
  __syncthreads();
  int gt_before = s_base[0] + (excl >> 16), eq_before = s_base[1] + (excl & 0xffff);
  int32_t* out = idx_out + bh * k;
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    if (j0 + e < P) {
      if (kv[e] > T) {
        out[gt_before + min(eq_before, remaining)] = j0 + e;
        ++gt_before;
      } else if (kv[e] == T) {
        if (eq_before < remaining) out[gt_before + eq_before] = j0 + e;
        ++eq_before;
      }
    }
  }
  cl.barrier_wait();  // no block leaves while another may still read its counts
}

// ---------------------------------------------------------------------------
// Eq. 4: the softmax-mass score S(j) = sum_r softmax_j(alpha q_r . k_j) over
// the rows r = (query head i of the group, proxy t), r = i * n_proxy + t,
// the softmax taken over the L current keys and S kept for j < P.
// Pass 1 (mass_stats_kernel): per key split (at most 32), each row's running maximum m
// and sum l of 2^(t - m), t = fl(z c), z = q_r . k_j (exact BF16 products,
// float32 accumulation: tcgen05 MMAs into tensor memory), c = alpha log2 e.
// Pass 2 (mass_colsum_kernel): the splits' partials merged per row (m = max
// over splits, l = sum_s l_s 2^(m_s - m), 1/l), then per 128-key tile of
// [0, P) the column sums of 2^(t - m) (1/l) over a group of at most 256
// rows; with one row group they are written as the order-preserving keys of
// the top-k kernels, else (mass_keys_kernel) the row groups' sums are added
// in a fixed order first.  Both passes stream the keys
// by TMA (128-byte swizzled tiles of the caller's BF16 cache) through a
// three-stage ring; one thread issues the MMAs into two TMEM buffers, so a
// tile's products run while the consumers read the previous one.
constexpr int kMassGroupRows = 256;   // rows of one row group (two M = 128 halves)
constexpr int kMassSplits = 32;       // most key splits of pass 1 per (sequence, KV head, row group)
constexpr int kMassTileKeys = 128;    // keys per tile (MMA N in pass 1, M in pass 2)
constexpr int kMassCons = 256;        // consumer threads (warps 0-7)
constexpr int kMassTmaWarp = 8, kMassMmaWarp = 9;
constexpr int kMassThreads = 320;
constexpr int kMassStages = 4;        // key-tile ring
constexpr uint32_t kMassTmemCols = 512;
// Shared memory from a 1024-byte aligned base.  Operand images are K-major
// (dims contiguous) in the 128-byte-swizzled layout, one region per 64
// dims: the row group's queries [dim half][256 rows][128 B], each key stage
// [dim half][128 keys][128 B].
constexpr int kMOffQ = 0;
constexpr int kMQHalf = kMassGroupRows * 128;          // 32 KB
constexpr int kMKHalf = kMassTileKeys * 128;           // 16 KB
constexpr int kMOffK = kMOffQ + 2 * kMQHalf;
constexpr int kMOffSt = kMOffK + kMassStages * 2 * kMKHalf;  // pass 2: (-m, 1/l) of row pairs, float4 [128]
constexpr int kMOffX = kMOffSt + 128 * 16;                   // pass 2: column-sum exchange, float [2][128]
constexpr int kMOffBar = kMOffX + 2 * 128 * 4;
constexpr int kMOffMisc = kMOffBar + 16 * 8;
constexpr int kMassSmem = kMOffMisc + 64 + 1024;        // + room to align the base

// Shared-memory load by address (a warp reading one address is one broadcast).
__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];\n" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ float mass_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct MassParams {
  const __nv_bfloat16* qp;  // [B][HQ][n_ld][128]
  int32_t n_proxy, n_ld, gq, R, n_groups;
  int32_t L;      // pass 1: keys [0, L); pass 2: column sums of [0, L) (= P)
  int32_t ld;     // rows per (sequence, KV head) in the key source
  float c;        // fl(alpha log2 e)
  int32_t q_tma;         // the row group's query rows are contiguous: loaded by TMA
  float2* part;          // pass 1 output, pass 2 input
  int32_t ns;            // pass 1 splits
  float* colsum;         // pass 2 output with more than one row group
  uint32_t* keys;        // pass 2 output with one row group: the top-k keys
  int32_t pmax;
  int32_t* err;
};

// 2D tiled load of a box of 64 dims x rows (128-byte swizzle) from a BF16
// source viewed as [rows][128 dims]; completion counted on `bar`.
__device__ __forceinline__ void tma_load_k(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// The row group's queries -> the swizzled K-major image (rows past R zero),
// by every thread of the block, made visible to the tensor core.
__device__ void mass_stage_q_tc(uint8_t* sm, const MassParams& p, int b, int h, int HKV, int rg) {
  // all of a thread's loads are issued before its first store
  constexpr int kPer = (kMassGroupRows * 16 + kMassThreads - 1) / kMassThreads;
  uint4 v[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = threadIdx.x + u * kMassThreads, lr = i >> 4, c = i & 15, r = rg * kMassGroupRows + lr;
    v[u] = make_uint4(0, 0, 0, 0);
    if (i < kMassGroupRows * 16 && r < p.R) {
      const int hi = r / p.n_proxy, t = r - hi * p.n_proxy;
      v[u] = __ldg(reinterpret_cast<const uint4*>(
                       p.qp + (((size_t)b * HKV * p.gq + (size_t)h * p.gq + hi) * p.n_ld + t) * HYQ_D) +
                   c);
    }
  }
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = threadIdx.x + u * kMassThreads, lr = i >> 4, c = i & 15;
    if (i < kMassGroupRows * 16)
      *reinterpret_cast<uint4*>(sm + kMOffQ + (c >> 3) * kMQHalf + lr * 128 + (((c & 7) ^ (lr & 7)) << 4)) = v[u];
  }
  fence_proxy_async_smem();
}

// Key tiles of one block: `n` tiles, tile i at key row `row0 + i * stride * 128`
// (rows of the flattened [B][HKV][ld] key source).  The loader thread of the
// TMA warp fills the ring, the MMA thread issues one tile's products into
// TMEM buffer i % 2 and releases the stage, the consumers read the buffer and
// release it.  kCols: TMEM columns per tile (pass 1: 2 x 128, pass 2: 256).
struct MassBars {
  uint64_t *kfull, *kempty, *dfull, *dfree, *mmadone, *qfull;
};

__device__ __forceinline__ MassBars mass_bars(uint8_t* sm) {
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kMOffBar);
  return MassBars{bars, bars + kMassStages, bars + 2 * kMassStages, bars + 2 * kMassStages + 2,
                  bars + 2 * kMassStages + 4, bars + 2 * kMassStages + 5};
}

__device__ void mass_init_bars(const MassBars& mb) {
  for (int i = 0; i < kMassStages; ++i) {
    mbar_init(mb.kfull + i, 1);
    mbar_init(mb.kempty + i, 1);
  }
  for (int i = 0; i < 2; ++i) {
    mbar_init(mb.dfull + i, 1);
    mbar_init(mb.dfree + i, kMassCons);
  }
  mbar_init(mb.mmadone, 1);
  mbar_init(mb.qfull, 1);
  mbar_fence_init();
}

// TMA warp, lane 0, at entry: the row group's 256 query rows (two 32 KB
// boxes) when they are contiguous in the proxy buffer.
__device__ void mass_load_q(uint8_t* sm, const MassBars& mb, const CUtensorMap* qmap, const MassParams& p, int b, int h,
                            int HKV, int rg) {
  const int y = (int)(((int64_t)b * HKV * p.gq + (int64_t)h * p.gq) * p.n_ld) + rg * kMassGroupRows;
  mbar_arrive_expect_tx(mb.qfull, 2 * kMQHalf);
  tma_load_k(sm + kMOffQ, qmap, 0, y, mb.qfull);
  tma_load_k(sm + kMOffQ + kMQHalf, qmap, 64, y, mb.qfull);
}

// TMA warp, lane 0: tiles [i0, i1) (the first kMassStages need no free
// stage and are issued at kernel entry, before the queries are staged).
__device__ void mass_loader(uint8_t* sm, const MassBars& mb, const CUtensorMap* map, int i0, int i1, int64_t row0,
                            int64_t stride, volatile int* abort_flag, int32_t* err) {
  int last = i0 - 1;
  bool ok = true;
  for (int i = i0; i < i1; ++i) {
    const int s = i % kMassStages;
    if (i >= kMassStages && !mbar_wait_or_abort(mb.kempty + s, ((i / kMassStages) & 1) ^ 1, abort_flag)) {
      ok = false;
      break;
    }
    uint8_t* dst = sm + kMOffK + s * 2 * kMKHalf;
    const int y = (int)(row0 + (int64_t)i * stride * kMassTileKeys);
    mbar_arrive_expect_tx(mb.kfull + s, 2 * kMKHalf);
    tma_load_k(dst, map, 0, y, mb.kfull + s);
    tma_load_k(dst + kMKHalf, map, 64, y, mb.kfull + s);
    last = i;
  }
  if (!ok) {
    *abort_flag = 1;
    hyq_set_err(err, HYQ_DEVERR_TIMEOUT);
    // the copies in flight land before the block's shared memory goes away
    for (int i = max(0, last - kMassStages + 1); i <= last; ++i)
      (void)mbar_wait(mb.kfull + i % kMassStages, (i / kMassStages) & 1);
  }
}

// MMA warp, lane 0.  kPass2: D[key][row] = K Q^T (M = 128 keys, N = 256
// rows); else D_h[row][key] = Q_h K^T for the row halves h (M = 128, N = 128).
template <bool kPass2>
__device__ void mass_mma(uint8_t* sm, const MassBars& mb, uint32_t tbase, int n, bool q_tma, volatile int* abort_flag,
                         int32_t* err) {
  constexpr uint32_t kIdesc = tc_idesc(kTcBF16, kTcBF16, 128, kPass2 ? 256 : 128);
  const uint64_t dQ = tc_desc_sw128(smem_u32(sm + kMOffQ)), dK0 = tc_desc_sw128(smem_u32(sm + kMOffK));
  bool ok = !(q_tma && n > 0) || mbar_wait_or_abort(mb.qfull, 0, abort_flag);
  for (int i = 0; ok && i < n; ++i) {
    const int s = i % kMassStages, bf = i & 1;
    ok = mbar_wait_or_abort(mb.kfull + s, (i / kMassStages) & 1, abort_flag);
    if (ok && i >= 2) ok = mbar_wait_or_abort(mb.dfree + bf, ((i >> 1) & 1) ^ 1, abort_flag);
    if (!ok) break;
    tc_fence_after();
    const uint64_t dK = dK0 + (uint64_t)(s * 2 * kMKHalf >> 4);
    const uint32_t tD = tbase + bf * 256;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      // 16 dims = 32 bytes per step; dims 64.. in the second region
      const uint64_t kq = (uint64_t)((ks >> 2) * kMQHalf >> 4) + (ks & 3) * 2;
      const uint64_t kk = (uint64_t)((ks >> 2) * kMKHalf >> 4) + (ks & 3) * 2;
      if (kPass2) {
        tc_mma_f16(tD, dK + kk, dQ + kq, kIdesc, ks > 0);
      } else {
        tc_mma_f16(tD, dQ + kq, dK + kk, kIdesc, ks > 0);
        tc_mma_f16(tD + 128, dQ + kq + (kMKHalf >> 4), dK + kk, kIdesc, ks > 0);  // rows 128..255
      }
    }
    tc_commit(mb.dfull + bf);
    tc_commit(mb.kempty + s);
  }
  if (!ok) {
    *abort_flag = 1;
    hyq_set_err(err, HYQ_DEVERR_TIMEOUT);
  }
  tc_commit(mb.mmadone);  // every MMA issued has finished once this arrives
  (void)mbar_wait(mb.mmadone, 0);
}

// Consumer: the 128 FP32 columns [col, col + 128) of this thread's TMEM lane.
__device__ __forceinline__ void mass_ld128(uint32_t taddr, float (&x)[128]) {
  uint32_t r[4][32];
#pragma unroll
  for (int c = 0; c < 4; ++c) tc_ld32(taddr + 32 * c, r[c]);
  tc_wait_ld();
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int i = 0; i < 32; ++i) x[32 * c + i] = __uint_as_float(r[c][i]);
}

// Pass 1.  grid (splits <= kMassSplits, HKV * n_groups, B), 320 threads.
// Split s takes the 128-key tiles [s nt / S, (s + 1) nt / S) of [0, L);
// consumer thread = row (TMEM lane) of one row half: per tile the maximum
// of t = fl(z c) and the running (m, l), l the sum of ex2(fl(z c - m)).
// part[((bh * n_groups + rg) * kMassSplits + split) * 256 + row] = (m, l).
__global__ void __launch_bounds__(kMassThreads, 1)
    mass_stats_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ MassParams p) {
  extern __shared__ uint8_t mass_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(mass_raw) + 1023) & ~(uintptr_t)1023);
  const MassBars mb = mass_bars(sm);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + kMOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kMOffMisc + 4);
  const int split = blockIdx.x, ns = gridDim.x, HKV = gridDim.y / p.n_groups;
  const int h = blockIdx.y / p.n_groups, rg = blockIdx.y % p.n_groups, b = blockIdx.z;
  const size_t bh = (size_t)b * HKV + h;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = (p.L + kMassTileKeys - 1) / kMassTileKeys;
  const int t0 = (int)((int64_t)split * nt / ns), t1 = (int)((int64_t)(split + 1) * nt / ns);
  const int n = t1 - t0;
  const int64_t krow0 = (int64_t)bh * p.ld + (int64_t)t0 * kMassTileKeys;
  const int nprime = min(n, kMassStages);
  if (threadIdx.x == kMassTmaWarp * 32) {
    mass_init_bars(mb);
    *abort_flag = 0;
    if (p.q_tma && n > 0) mass_load_q(sm, mb, &qmap, p, b, h, HKV, rg);
    mass_loader(sm, mb, &kmap, 0, nprime, krow0, 1, abort_flag, p.err);
  }
  if (!p.q_tma) mass_stage_q_tc(sm, p, b, h, HKV, rg);
  if (warp == kMassMmaWarp) tc_alloc(tslot, kMassTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp < 8) {
    const int half = warp >> 2, row = 128 * half + 32 * (warp & 3) + lane;
    const uint32_t tl = tbase + ((uint32_t)(32 * (warp & 3)) << 16) + 128 * half;
    const uint64_t c2 = f2_splat(p.c);
    float m = -INFINITY, l = 0.f;
    for (int i = 0; i < n; ++i) {
      const int bf = i & 1;
      if (!mbar_wait_or_abort(mb.dfull + bf, (i >> 1) & 1, abort_flag)) {
        *abort_flag = 1;
        hyq_set_err(p.err, HYQ_DEVERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      float x[128];
      mass_ld128(tl + bf * 256, x);
      tc_fence_before();
      mbar_arrive(mb.dfree + bf);
      const int nvalid = p.L - (t0 + i) * kMassTileKeys;  // keys of the tile inside [0, L)
      // keys past L are -inf
      if (nvalid < kMassTileKeys) {
#pragma unroll
        for (int k = 0; k < 128; ++k) x[k] = k < nvalid ? x[k] : -INFINITY;
      }
      // the tile maximum of t = fl(z c) is fl(max z * c) (c > 0, rounding
      // is monotone)
      float a[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) a[u] = -INFINITY;
#pragma unroll
      for (int k = 0; k < 64; ++k) a[k & 7] = fmax3(a[k & 7], x[2 * k], x[2 * k + 1]);
      const float zm = fmax3(fmax3(a[0], a[1], a[2]), fmax3(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
      const float tm = zm == -INFINITY ? -INFINITY : zm * p.c;
      const float mn = fmaxf(m, tm);
      if (mn != -INFINITY) {
        // ex2 of fl(z c - m): one rounding where fl(fl(z c) - m) has two
        const uint64_t nm2 = f2_splat(-mn);
        uint64_t s2[4] = {0, 0, 0, 0};
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          const uint64_t d2 = f2_fma(f2_pack(x[2 * k], x[2 * k + 1]), c2, nm2);
          s2[k & 3] = f2_add(s2[k & 3], f2_pack(mass_ex2(f2_lo(d2)), mass_ex2(f2_hi(d2))));
        }
        const uint64_t r2 = f2_add(f2_add(s2[0], s2[1]), f2_add(s2[2], s2[3]));
        l = l * mass_ex2(m - mn) + (f2_lo(r2) + f2_hi(r2));
        m = mn;
      }
    }
    p.part[((bh * p.n_groups + rg) * kMassSplits + split) * kMassGroupRows + row] = make_float2(m, l);
  } else if (warp == kMassTmaWarp) {
    if (lane == 0) {
      mass_loader(sm, mb, &kmap, nprime, n, krow0, 1, abort_flag, p.err);
      if (p.q_tma && n > 0) (void)mbar_wait(mb.qfull, 0);  // the query copy has landed (also after a failure)
    }
  } else if (lane == 0) {
    mass_mma<false>(sm, mb, tbase, n, p.q_tma != 0, abort_flag, p.err);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMassMmaWarp) {
    tc_fence_after();
    tc_dealloc(tbase, kMassTmemCols);
  }
}

// Pass 2.  grid (blocks, HKV * n_groups, B), 320 threads; block x takes the
// 128-key tiles x, x + blocks, ... of [0, P).  D = K Q^T puts a key in each
// TMEM lane and the group's 256 rows in the columns; consumer warp w takes
// the keys of lane quarter w % 4 and the rows 128 (w / 4) .. + 127: the sum
// over its rows of fma(ex2(fl(z c - m_r)), 1 / l_r); the two row halves are
// added in a fixed order.  colsum[(bh * n_groups + rg) * pmax + j].
__global__ void __launch_bounds__(kMassThreads, 1)
    mass_colsum_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                       const __grid_constant__ MassParams p) {
  extern __shared__ uint8_t mass_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(mass_raw) + 1023) & ~(uintptr_t)1023);
  const MassBars mb = mass_bars(sm);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + kMOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kMOffMisc + 4);
  float4* st4 = reinterpret_cast<float4*>(sm + kMOffSt);  // rows (2i, 2i+1): (-m, -m, 1/l, 1/l)
  float* xch = reinterpret_cast<float*>(sm + kMOffX);     // [2][128]
  const int HKV = gridDim.y / p.n_groups, h = blockIdx.y / p.n_groups, rg = blockIdx.y % p.n_groups;
  const int b = blockIdx.z;
  const size_t bh = (size_t)b * HKV + h, bg = bh * p.n_groups + rg;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = (p.L + kMassTileKeys - 1) / kMassTileKeys;
  const int n = (int)blockIdx.x < nt ? (nt - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int64_t krow0 = (int64_t)bh * p.ld + (int64_t)blockIdx.x * kMassTileKeys;
  const int nprime = min(n, kMassStages);
  if (threadIdx.x == kMassTmaWarp * 32) {
    mass_init_bars(mb);
    *abort_flag = 0;
    if (p.q_tma && n > 0) mass_load_q(sm, mb, &qmap, p, b, h, HKV, rg);
    mass_loader(sm, mb, &kmap, 0, nprime, krow0, gridDim.x, abort_flag, p.err);
  }
  if (!p.q_tma) mass_stage_q_tc(sm, p, b, h, HKV, rg);
  if (warp == kMassMmaWarp) tc_alloc(tslot, kMassTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp < 8) {
    {
      // Row r's split partials merged: m the largest, l the sum over splits
      // (in split order) of l_s 2^(m_s - m), and 1/l; rows past R weigh 0.
      const int r = threadIdx.x;
      float mr = 0.f, il = 0.f;
      if (rg * kMassGroupRows + r < p.R) {
        const float2* pr = p.part + bg * kMassSplits * kMassGroupRows + r;
        float2 v[kMassSplits];
#pragma unroll
        for (int q = 0; q < kMassSplits; ++q) v[q] = q < p.ns ? pr[q * kMassGroupRows] : make_float2(-INFINITY, 0.f);
        float mx = -INFINITY;
#pragma unroll
        for (int q = 0; q < kMassSplits; ++q) mx = fmaxf(mx, v[q].x);
        float l = 0.f;
        if (mx != -INFINITY) {
#pragma unroll
          for (int q = 0; q < kMassSplits; ++q)
            if (v[q].x != -INFINITY) l += v[q].y * mass_ex2(v[q].x - mx);
        }
        mr = mx == -INFINITY ? 0.f : mx;
        il = l > 0.f ? __frcp_rn(l) : 0.f;
      }
      float* sf = reinterpret_cast<float*>(st4);
      sf[(r >> 1) * 4 + (r & 1)] = -mr;
      sf[(r >> 1) * 4 + 2 + (r & 1)] = il;
    }
    asm volatile("bar.sync 1, 256;\n" ::: "memory");  // the rows' constants are in shared memory
    const int half = warp >> 2, key = 32 * (warp & 3) + lane;
    const uint32_t tl = tbase + ((uint32_t)(32 * (warp & 3)) << 16) + 128 * half;
    const uint32_t sth = smem_u32(st4 + 64 * half);
    const uint64_t c2 = f2_splat(p.c);
    // Every consumer runs all n iterations (the named barrier below is
    // passed once per tile by all 256); after a failed wait a thread skips
    // the work of the remaining tiles.
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      const int bf = i & 1;
      const int j0 = ((int)blockIdx.x + i * (int)gridDim.x) * kMassTileKeys;
      if (ok && !mbar_wait_or_abort(mb.dfull + bf, (i >> 1) & 1, abort_flag)) {
        *abort_flag = 1;
        hyq_set_err(p.err, HYQ_DEVERR_TIMEOUT);
        ok = false;
      }
      float cs = 0.f;
      if (ok) {
        tc_fence_after();
        float x[128];
        mass_ld128(tl + bf * 256, x);
        tc_fence_before();
        mbar_arrive(mb.dfree + bf);
        uint64_t acc2[2] = {0, 0};
#pragma unroll
        for (int k = 0; k < 64; ++k) {  // rows 128 half + 2k, + 2k + 1
          const float4 s = lds_f4(sth + 16 * k);
          const uint64_t t2 = f2_fma(f2_pack(x[2 * k], x[2 * k + 1]), c2, f2_pack(s.x, s.y));  // fl(z c - m)
          const uint64_t e2 = f2_pack(mass_ex2(f2_lo(t2)), mass_ex2(f2_hi(t2)));
          acc2[k & 1] = f2_fma(e2, f2_pack(s.z, s.w), acc2[k & 1]);
        }
        const uint64_t r2 = f2_add(acc2[0], acc2[1]);
        cs = f2_lo(r2) + f2_hi(r2);
      }
      float* xb = xch + bf * 128;
      if (half) xb[key] = cs;
      asm volatile("bar.sync 1, 256;\n" ::: "memory");
      if (ok && !half && j0 + key < p.L) {
        const float S = cs + xb[key];
        if (p.keys)
          p.keys[bh * p.pmax + j0 + key] = order_key(S, p.err);
        else
          p.colsum[bg * p.pmax + j0 + key] = S;
      }
    }
  } else if (warp == kMassTmaWarp) {
    if (lane == 0) {
      mass_loader(sm, mb, &kmap, nprime, n, krow0, gridDim.x, abort_flag, p.err);
      if (p.q_tma && n > 0) (void)mbar_wait(mb.qfull, 0);  // the query copy has landed (also after a failure)
    }
  } else if (lane == 0) {
    mass_mma<true>(sm, mb, tbase, n, p.q_tma != 0, abort_flag, p.err);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMassMmaWarp) {
    tc_fence_after();
    tc_dealloc(tbase, kMassTmemCols);
  }
}

// Final.  grid (ceil(P / 256), HKV, B): S(j) = sum over row groups (fixed
// order) -> order-preserving key.
__global__ void mass_keys_kernel(const float* __restrict__ colsum, int32_t n_groups, int32_t P, int32_t pmax,
                                 uint32_t* __restrict__ keys, int32_t* err) {
  const size_t bh = (size_t)blockIdx.z * gridDim.y + blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= P) return;
  float S = 0.f;
  for (int rg = 0; rg < n_groups; ++rg) S += colsum[(bh * n_groups + rg) * pmax + j];
  keys[bh * pmax + j] = order_key(S, err);
}

}  // namespace

size_t hyq_select_kv_ws_bytes(const hyq_config* c, int32_t L) {
  size_t bh = (size_t)c->batch * c->num_kv_heads;
  int32_t P = L - c->window > 0 ? L - c->window : 0;
  return 256 + round_up(bh * HYQ_D * 4) + round_up(bh * (size_t)(P > 0 ? P : 1) * 4);
}

size_t hyq_select_ws_bytes(const hyq_config* c, int32_t L) {
  const size_t kv = hyq_select_kv_ws_bytes(c, L);
  if (c->vl_mode != HYQ_VL_PER_QUERY_HEAD) return kv;
  const size_t bq = (size_t)c->batch * c->num_q_heads;
  const int32_t P = L - c->window > 0 ? L - c->window : 0;
  const size_t k1 = (size_t)hyq_vl_count_head(c, P);
  return kv + round_up(bq * HYQ_D * 4) + round_up(bq * (size_t)(P > 0 ? P : 1) * 4) +
         round_up(bq * (k1 > 0 ? k1 : 1) * 4);
}

namespace {

// Row groups of the mass score for n_proxy proxy rows per query head.
int32_t mass_groups(const hyq_config* c, int32_t n_proxy) {
  const int32_t R = c->num_q_heads / c->num_kv_heads * n_proxy;
  return (R + kMassGroupRows - 1) / kMassGroupRows;
}

struct MassWs {
  float2* part;    // [bh][groups][kMassSplits][256]
  float* colsum;   // [bh][groups][P] (more than one row group)
};

MassWs carve_mass(const hyq_config* c, int32_t L, void* ws) {
  const size_t bh = (size_t)c->batch * c->num_kv_heads;
  const size_t ng = (size_t)mass_groups(c, c->period);
  char* p = static_cast<char*>(ws) + hyq_select_ws_bytes(c, L);
  MassWs w;
  w.part = reinterpret_cast<float2*>(p);
  p += round_up(bh * ng * kMassSplits * kMassGroupRows * sizeof(float2));
  w.colsum = reinterpret_cast<float*>(p);
  return w;
}

// Top-k of `heads` rows of P keys per sequence ([B][heads][P]).
cudaError_t launch_topk_rows(const hyq_config* c, const uint32_t* keys, int32_t heads, int32_t P, int32_t k,
                             int32_t* idx_out, cudaStream_t s) {
  const int32_t cap = kTopkCluster * kTopkCtaThreads;
  dim3 gc(kTopkCluster, heads, c->batch);
  if (P <= 4 * cap) {
    topk_cluster_kernel<4><<<gc, kTopkCtaThreads, 0, s>>>(keys, P, P, k, idx_out);
    return cudaGetLastError();
  }
  if (P <= 8 * cap) {
    topk_cluster_kernel<8><<<gc, kTopkCtaThreads, 0, s>>>(keys, P, P, k, idx_out);
    return cudaGetLastError();
  }
  if (P <= 16 * cap) {
    topk_cluster_kernel<16><<<gc, kTopkCtaThreads, 0, s>>>(keys, P, P, k, idx_out);
    return cudaGetLastError();
  }
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t ea = hyq_once_per_device(attr_done, [] {
    return cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kTopkSmemKeys * (int)sizeof(uint32_t));
  });
  if (ea != cudaSuccess) return ea;
  const size_t tk_smem = P <= kTopkSmemKeys ? (size_t)P * sizeof(uint32_t) : 0;
  topk_kernel<<<dim3(heads, c->batch), kTopkThreads, tk_smem, s>>>(keys, P, P, k, idx_out);
  return cudaGetLastError();
}

cudaError_t launch_topk(const hyq_config* c, const SelectWs& w, int32_t P, int32_t k, int32_t* idx_out,
                        cudaStream_t s) {
  return launch_topk_rows(c, w.keys, c->num_kv_heads, P, k, idx_out, s);
}

// Per-query-head workspace, after the per-KV-head one: u per query head,
// keys per query head, the heads' index lists.
struct HeadsWs {
  float* u;
  uint32_t* keys;
  int32_t* idx;
};

HeadsWs carve_heads(const hyq_config* c, int32_t L, void* ws) {
  const size_t bq = (size_t)c->batch * c->num_q_heads;
  const int32_t P = L - c->window > 0 ? L - c->window : 0;
  char* p = static_cast<char*>(ws) + hyq_select_kv_ws_bytes(c, L);
  HeadsWs w;
  w.u = reinterpret_cast<float*>(p);
  p += round_up(bq * HYQ_D * 4);
  w.keys = reinterpret_cast<uint32_t*>(p);
  p += round_up(bq * (size_t)(P > 0 ? P : 1) * 4);
  w.idx = reinterpret_cast<int32_t*>(p);
  (void)P;
  return w;
}

}  // namespace

size_t hyq_select_mass_ws_bytes(const hyq_config* c, int32_t L) {
  const size_t bh = (size_t)c->batch * c->num_kv_heads;
  const size_t ng = (size_t)mass_groups(c, c->period);
  int32_t P = L - c->window > 0 ? L - c->window : 0;
  return hyq_select_ws_bytes(c, L) + round_up(bh * ng * kMassSplits * kMassGroupRows * sizeof(float2)) +
         round_up(bh * ng * (size_t)(P > 0 ? P : 1) * 4);
}

cudaError_t hyq_launch_select(const hyq_config* c, const void* q_proxy, int32_t n_proxy,
                              int32_t n_proxy_ld, const void* k_src, int32_t ld, int32_t L,
                              int32_t* idx_out, int32_t k, void* ws, cudaStream_t s) {
  SelectWs w = carve(c, L, ws);
  const int32_t P = L - c->window;  // > 0 since k > 0
  const int32_t gq = c->num_q_heads / c->num_kv_heads;
  proxy_sum_kernel<<<dim3(c->num_kv_heads, c->batch), kProxyThreads, 0, s>>>(
      static_cast<const __nv_bfloat16*>(q_proxy), n_proxy, n_proxy_ld, gq, w.u);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 g2((P + kScoreRowsPerCta - 1) / kScoreRowsPerCta, c->num_kv_heads, c->batch);
  score_kernel<<<g2, kScoreThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(k_src), ld, P, w.u,
                                            w.keys, P, w.err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_topk(c, w, P, k, idx_out, s);
}

namespace {

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tmap_encode() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// A BF16 source [rows][128] as a TMA map whose box is 64 dims x box_rows rows
// with the 128-byte swizzle of the tensor-core operands; rows past the end
// read as zero.
cudaError_t make_row_map(CUtensorMap* map, const void* src, uint64_t rows, uint32_t box_rows) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encode();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {HYQ_D, rows};
  const cuuint64_t strides[1] = {HYQ_D * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(src), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t hyq_launch_select_mass(const hyq_config* c, const void* q_proxy, int32_t n_proxy,
                                   int32_t n_proxy_ld, const void* k_src, int32_t ld, int32_t L,
                                   int32_t* idx_out, int32_t k, void* ws, cudaStream_t s) {
  SelectWs w = carve(c, L, ws);
  MassWs mw = carve_mass(c, L, ws);
  const int32_t P = L - c->window;  // > 0 since k > 0
  const int32_t gq = c->num_q_heads / c->num_kv_heads, R = gq * n_proxy, ng = mass_groups(c, n_proxy);
  const float cs = (float)(1.0 / std::sqrt((double)HYQ_D) / std::log(2.0));  // fl(alpha log2 e)
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t ea = hyq_once_per_device(attr_done, [&] {
    cudaError_t e = cudaFuncSetAttribute(mass_stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMassSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(mass_colsum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMassSmem);
    return e;
  });
  if (ea != cudaSuccess) return ea;
  CUtensorMap kmap, qmap;
  cudaError_t e = make_row_map(&kmap, k_src, (uint64_t)c->batch * c->num_kv_heads * (uint64_t)ld, kMassTileKeys);
  if (e == cudaSuccess)
    e = make_row_map(&qmap, q_proxy, (uint64_t)c->batch * c->num_q_heads * (uint64_t)n_proxy_ld, kMassGroupRows);
  if (e != cudaSuccess) return e;
  // one block per SM (a block holds all 512 TMEM columns): the key tiles of a
  // (sequence, KV head, row group) are shared by floor(SMs / units) blocks
  const int n_sm = hyq_num_sms();
  const int units = c->num_kv_heads * ng * c->batch;
  const int per = std::max(1, n_sm / units);
  const int nt1 = (L + kMassTileKeys - 1) / kMassTileKeys, ntp = (P + kMassTileKeys - 1) / kMassTileKeys;
  const int ns = std::max(1, std::min({kMassSplits, per, nt1}));
  const int ncol = std::max(1, std::min(per, ntp));
  MassParams mp{};
  mp.qp = static_cast<const __nv_bfloat16*>(q_proxy);
  mp.n_proxy = n_proxy;
  mp.n_ld = n_proxy_ld;
  mp.gq = gq;
  mp.R = R;
  mp.n_groups = ng;
  mp.L = L;
  mp.ld = ld;
  mp.c = cs;
  // every row group is 256 rows contiguous in the proxy buffer: TMA
  mp.q_tma = (n_proxy == n_proxy_ld && R % kMassGroupRows == 0) ? 1 : 0;
  mp.part = mw.part;
  mp.ns = ns;
  mp.colsum = mw.colsum;
  mp.keys = ng == 1 ? w.keys : nullptr;  // one row group: pass 2 writes the keys itself
  mp.pmax = P;
  mp.err = w.err;
  mass_stats_kernel<<<dim3(ns, c->num_kv_heads * ng, c->batch), kMassThreads, kMassSmem, s>>>(kmap, qmap, mp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mp.L = P;
  mass_colsum_kernel<<<dim3(ncol, c->num_kv_heads * ng, c->batch), kMassThreads, kMassSmem, s>>>(kmap, qmap, mp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (ng > 1) {
    mass_keys_kernel<<<dim3((P + 255) / 256, c->num_kv_heads, c->batch), 256, 0, s>>>(mw.colsum, ng, P, P, w.keys,
                                                                                     w.err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return launch_topk(c, w, P, k, idx_out, s);
}

cudaError_t hyq_launch_select_heads(const hyq_config* c, const void* q_proxy, int32_t n_proxy,
                                    int32_t n_proxy_ld, const void* k_src, int32_t ld, int32_t L,
                                    int32_t* idx_heads, int32_t k1, int32_t* idx_out, int32_t ku, void* ws,
                                    cudaStream_t s) {
  SelectWs w = carve(c, L, ws);
  HeadsWs hw = carve_heads(c, L, ws);
  if (!idx_heads) idx_heads = hw.idx;
  const int32_t P = L - c->window;  // > 0 since k1 > 0
  const int32_t g = c->num_q_heads / c->num_kv_heads;
  const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(q_proxy);
  proxy_sum_kernel<<<dim3(c->num_q_heads, c->batch), kProxyThreads, 0, s>>>(qp, n_proxy, n_proxy_ld, 1, hw.u);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  proxy_sum_kernel<<<dim3(c->num_kv_heads, c->batch), kProxyThreads, 0, s>>>(qp, n_proxy, n_proxy_ld, g, w.u);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 g2((P + kScoreRowsPerCta - 1) / kScoreRowsPerCta, c->num_kv_heads, c->batch);
  const __nv_bfloat16* kk = static_cast<const __nv_bfloat16*>(k_src);
  switch (g) {
#define HYQ_SCORE_HEADS(G)                                                                                    \
  case G:                                                                                                    \
    score_heads_kernel<G><<<g2, kScoreThreads, 0, s>>>(kk, ld, P, hw.u, w.u, hw.keys, w.keys, w.err); \
    break;
    HYQ_SCORE_HEADS(1)
    HYQ_SCORE_HEADS(2)
    HYQ_SCORE_HEADS(3)
    HYQ_SCORE_HEADS(4)
    HYQ_SCORE_HEADS(5)
    HYQ_SCORE_HEADS(6)
    HYQ_SCORE_HEADS(7)
    HYQ_SCORE_HEADS(8)
#undef HYQ_SCORE_HEADS
    default:
      return cudaErrorInvalidValue;
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_topk_rows(c, hw.keys, c->num_q_heads, P, k1, idx_heads, s);
  if (e != cudaSuccess) return e;
  mark_union_kernel<<<dim3(c->num_q_heads, c->batch), 256, 0, s>>>(idx_heads, k1, g, P, w.keys);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_topk_rows(c, w.keys, c->num_kv_heads, P, ku, idx_out, s);
}
