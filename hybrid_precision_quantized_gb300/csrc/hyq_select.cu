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
  for (int r = r0; r < rows; r += 32) {
    const int j = r / n_proxy, t = r - j * n_proxy;
    const __nv_bfloat16* row = qp + (((size_t)b * HKV * gq + (size_t)h * gq + j) * n_ld + t) * HYQ_D;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(row) + c);
    const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(p2[i]);
      acc[2 * i] += f.x;
      acc[2 * i + 1] += f.y;
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
  for (int r0 = blockIdx.x * kScoreRowsPerCta + 2 * warp; r0 < end; r0 += 2 * (kScoreThreads / 32)) {
    const int r = r0 + half;
    const bool valid = r < end;
    float s[G + 1];
#pragma unroll
    for (int q = 0; q <= G; ++q) s[q] = 0.f;
    if (valid) {
      uint4 raw = *reinterpret_cast<const uint4*>(kb + (size_t)r * HYQ_D + 8 * sub);
      const __nv_bfloat162* pr = reinterpret_cast<const __nv_bfloat162*>(&raw);
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
// float32 accumulation on the tensor cores), c = alpha log2 e.  Merge
// (mass_merge_kernel): m = max over splits, l = sum_s l_s 2^(m_s - m), and
// 1/l.  Pass 2 (mass_colsum_kernel): per 64-key tile of [0, P), the column
// sums of 2^(t - m) (1/l) over a group of at most 256 rows.  Final
// (mass_keys_kernel): the row groups' sums in a fixed order, as the
// order-preserving keys of the top-k kernels.
constexpr int kMassThreads = 256;     // 8 warps, each two 16-row blocks of a row group
constexpr int kMassGroupRows = 256;
constexpr int kMassKeys = 64;         // keys per tile (8 MMA n-blocks)
constexpr int kMassStride = 136;      // bf16 per staged row: 272 bytes, conflict-free fragment loads
constexpr int kMassSplits = 32;       // most key splits of pass 1 per (sequence, KV head, row group)

__device__ __forceinline__ float mass_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Stage the query rows [rg * 256, +256) of the group into shared memory
// (stride kMassStride); rows past R are zero.
__device__ void mass_stage_q(__nv_bfloat16* qs, const __nv_bfloat16* qp, int b, int h, int HKV, int gq,
                             int n_proxy, int n_ld, int R, int rg) {
  for (int i = threadIdx.x; i < kMassGroupRows * 16; i += kMassThreads) {
    const int lr = i >> 4, c = i & 15, r = rg * kMassGroupRows + lr;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < R) {
      const int hi = r / n_proxy, t = r - hi * n_proxy;
      v = __ldg(reinterpret_cast<const uint4*>(qp + (((size_t)b * HKV * gq + (size_t)h * gq + hi) * n_ld + t) * HYQ_D) + c);
    }
    *reinterpret_cast<uint4*>(qs + lr * kMassStride + 8 * c) = v;
  }
}

// Start the asynchronous copy of key rows [j0, j0 + 64) of (b, h) into a
// staging buffer (rows past `end` are zero-filled) and commit it as one
// group of this thread's copies.
__device__ void mass_stage_k_async(__nv_bfloat16* ks, const __nv_bfloat16* kb, int j0, int end) {
  for (int i = threadIdx.x; i < kMassKeys * 16; i += kMassThreads) {
    const int r = i >> 4, c = i & 15;
    const bool in = j0 + r < end;
    const __nv_bfloat16* src = kb + (size_t)(in ? j0 + r : 0) * HYQ_D + 8 * c;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(ks + r * kMassStride + 8 * c)),
                 "l"(src), "r"(in ? 16 : 0)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}

// Wait until at most `n` of this thread's most recent copy groups are pending.
template <int n>
__device__ __forceinline__ void mass_wait_async() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(n) : "memory");
}

// A fragments (m16n8k16, row-major 16 x 128) of the 16-row block rb.
__device__ __forceinline__ void mass_load_a(const __nv_bfloat16* qs, int rb, int lane, uint32_t (&a)[8][4]) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t* r0 = reinterpret_cast<const uint32_t*>(qs + (16 * rb + g) * kMassStride + 16 * ks + 2 * t);
    const uint32_t* r8 = reinterpret_cast<const uint32_t*>(qs + (16 * rb + g + 8) * kMassStride + 16 * ks + 2 * t);
    a[ks][0] = r0[0];
    a[ks][1] = r8[0];
    a[ks][2] = r0[4];
    a[ks][3] = r8[4];
  }
}

// z = Q K^T for the warp's two row blocks and the staged 64-key tile:
// C[blk][nb][i] is row 16 rb + g + 8 (i >> 1), key 8 nb + 2 t + (i & 1).
__device__ __forceinline__ void mass_tile(const __nv_bfloat16* ksm, int lane, const uint32_t (&a0)[8][4],
                                          const uint32_t (&a1)[8][4], float (&C)[2][8][4]) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int blk = 0; blk < 2; ++blk)
#pragma unroll
    for (int nb = 0; nb < 8; ++nb) C[blk][nb][0] = C[blk][nb][1] = C[blk][nb][2] = C[blk][nb][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
#pragma unroll
    for (int nb = 0; nb < 8; ++nb) {
      const uint32_t* kr = reinterpret_cast<const uint32_t*>(ksm + (8 * nb + g) * kMassStride + 16 * ks + 2 * t);
      const uint32_t b0 = kr[0], b1 = kr[4];
      mma_bf16(C[0][nb], a0[ks], b0, b1);
      mma_bf16(C[1][nb], a1[ks], b0, b1);
    }
}

// Pass 1.  grid (splits <= kMassSplits, HKV * n_groups, B); dynamic smem: the row
// group's queries and two key tiles (one landing while the other is used).  part[((bh * n_groups + rg) *
// kMassSplits + split) * 256 + row] = (m, l) of the split's keys.
__global__ void __launch_bounds__(kMassThreads) mass_stats_kernel(
    const __nv_bfloat16* __restrict__ qp, int32_t n_proxy, int32_t n_ld, int32_t gq,
    const __nv_bfloat16* __restrict__ k_src, int32_t ld, int32_t L, float c, int32_t R, int32_t n_groups,
    float2* __restrict__ part) {
  extern __shared__ __align__(16) unsigned char mass_smem[];
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(mass_smem);
  __nv_bfloat16* ksm = qs + kMassGroupRows * kMassStride;
  const int split = blockIdx.x, HKV = gridDim.y / n_groups, h = blockIdx.y / n_groups, rg = blockIdx.y % n_groups;
  const int b = blockIdx.z;
  const size_t bh = (size_t)b * HKV + h;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = lane & 3;
  mass_stage_q(qs, qp, b, h, HKV, gq, n_proxy, n_ld, R, rg);
  __syncthreads();
  uint32_t a0[8][4], a1[8][4];
  mass_load_a(qs, 2 * warp, lane, a0);
  mass_load_a(qs, 2 * warp + 1, lane, a1);
  // rows (blk, half): 16 (2 warp + blk) + g + 8 half
  float m[2][2], l[2][2];
#pragma unroll
  for (int blk = 0; blk < 2; ++blk) m[blk][0] = m[blk][1] = -INFINITY, l[blk][0] = l[blk][1] = 0.f;
  const int ns = gridDim.x;
  const int j0 = (int)((int64_t)split * L / ns), j1 = (int)((int64_t)(split + 1) * L / ns);
  const __nv_bfloat16* kb = k_src + bh * ld * HYQ_D;
  // two staging buffers: tile i + 1 is in flight while tile i is consumed
  if (j0 < j1) mass_stage_k_async(ksm, kb, j0, j1);
  for (int kt = j0, it = 0; kt < j1; kt += kMassKeys, ++it) {
    __nv_bfloat16* kcur = ksm + (it & 1) * kMassKeys * kMassStride;
    if (kt + kMassKeys < j1) {
      mass_stage_k_async(ksm + ((it + 1) & 1) * kMassKeys * kMassStride, kb, kt + kMassKeys, j1);
      mass_wait_async<1>();
    } else {
      mass_wait_async<0>();
    }
    __syncthreads();  // tile `it` has landed for every thread
    float C[2][8][4];
    mass_tile(kcur, lane, a0, a1, C);
    const int nvalid = min(kMassKeys, j1 - kt);
#pragma unroll
    for (int blk = 0; blk < 2; ++blk)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float v[16];
        float tm = -INFINITY;
#pragma unroll
        for (int nb = 0; nb < 8; ++nb)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int key = 8 * nb + 2 * t + e;
            const float x = key < nvalid ? C[blk][nb][2 * hf + e] * c : -INFINITY;
            v[2 * nb + e] = x;
            tm = fmaxf(tm, x);
          }
        tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 1));
        tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 2));
        const float mn = fmaxf(m[blk][hf], tm);
        float sum = 0.f;
        if (mn != -INFINITY) {
#pragma unroll
          for (int i = 0; i < 16; ++i) sum += mass_ex2(v[i] - mn);
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        if (mn != -INFINITY) {
          l[blk][hf] = l[blk][hf] * mass_ex2(m[blk][hf] - mn) + sum;
          m[blk][hf] = mn;
        }
      }
    __syncthreads();  // every warp is done with buffer `it & 1` before it is refilled
  }
  if (t == 0) {
    float2* out = part + ((bh * n_groups + rg) * kMassSplits + split) * kMassGroupRows;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) out[16 * (2 * warp + blk) + (lane >> 2) + 8 * hf] = make_float2(m[blk][hf], l[blk][hf]);
  }
}

// Merge.  grid (HKV * n_groups, B), 256 threads (one row each):
// stats = (m, 1/l) over all splits; padding rows (past R) get weight 0.
__global__ void __launch_bounds__(kMassGroupRows) mass_merge_kernel(const float2* __restrict__ part,
                                                                    float2* __restrict__ stats, int32_t R,
                                                                    int32_t n_groups, int32_t ns) {
  const size_t bg = (size_t)blockIdx.y * gridDim.x + blockIdx.x;  // (bh, rg) flattened
  const int r = threadIdx.x;
  if ((int)(blockIdx.x % n_groups) * kMassGroupRows + r >= R) {
    stats[bg * kMassGroupRows + r] = make_float2(0.f, 0.f);
    return;
  }
  const float2* p = part + bg * kMassSplits * kMassGroupRows + r;
  float m = -INFINITY;
  for (int s = 0; s < ns; ++s) m = fmaxf(m, p[s * kMassGroupRows].x);
  float l = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < ns; ++s) {
      const float2 v = p[s * kMassGroupRows];
      if (v.x != -INFINITY) l += v.y * mass_ex2(v.x - m);
    }
  }
  stats[bg * kMassGroupRows + r] = make_float2(m == -INFINITY ? 0.f : m, l > 0.f ? __frcp_rn(l) : 0.f);
}

// Pass 2.  grid (blocks, HKV * n_groups, B), block x taking the 64-key tiles
// x, x + blocks, ... of [0, P): the row group's column sums of 2^(t - m) / l,
// in a fixed order.
// colsum[((bh * n_groups + rg) * pmax + j].
__global__ void __launch_bounds__(kMassThreads) mass_colsum_kernel(
    const __nv_bfloat16* __restrict__ qp, int32_t n_proxy, int32_t n_ld, int32_t gq,
    const __nv_bfloat16* __restrict__ k_src, int32_t ld, int32_t P, float c, int32_t R, int32_t n_groups,
    const float2* __restrict__ stats, float* __restrict__ colsum, int32_t pmax) {
  extern __shared__ __align__(16) unsigned char mass_smem[];
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(mass_smem);
  __nv_bfloat16* ksm = qs + kMassGroupRows * kMassStride;
  float* red = reinterpret_cast<float*>(ksm + 2 * kMassKeys * kMassStride);  // [8 warps][64 keys]
  const int HKV = gridDim.y / n_groups, h = blockIdx.y / n_groups, rg = blockIdx.y % n_groups;
  const int b = blockIdx.z;
  const size_t bh = (size_t)b * HKV + h, bg = bh * n_groups + rg;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  mass_stage_q(qs, qp, b, h, HKV, gq, n_proxy, n_ld, R, rg);
  __syncthreads();
  uint32_t a0[8][4], a1[8][4];
  mass_load_a(qs, 2 * warp, lane, a0);
  mass_load_a(qs, 2 * warp + 1, lane, a1);
  float2 st[2][2];  // this thread's rows: (m, 1/l)
#pragma unroll
  for (int blk = 0; blk < 2; ++blk)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) st[blk][hf] = stats[bg * kMassGroupRows + 16 * (2 * warp + blk) + g + 8 * hf];
  const __nv_bfloat16* kb = k_src + bh * ld * HYQ_D;
  const int step = gridDim.x * kMassKeys;
  if ((int)blockIdx.x * kMassKeys < P) mass_stage_k_async(ksm, kb, blockIdx.x * kMassKeys, P);
  for (int kt = blockIdx.x * kMassKeys, it = 0; kt < P; kt += step, ++it) {
  __nv_bfloat16* kcur = ksm + (it & 1) * kMassKeys * kMassStride;
  if (kt + step < P) {
    mass_stage_k_async(ksm + ((it + 1) & 1) * kMassKeys * kMassStride, kb, kt + step, P);
    mass_wait_async<1>();
  } else {
    mass_wait_async<0>();
  }
  __syncthreads();  // tile `it` has landed for every thread; the sums of the previous one are read
  float C[2][8][4];
  mass_tile(kcur, lane, a0, a1, C);
  float cs[8][2];
#pragma unroll
  for (int nb = 0; nb < 8; ++nb) cs[nb][0] = cs[nb][1] = 0.f;
#pragma unroll
  for (int blk = 0; blk < 2; ++blk)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)  // rows past R have 1/l = 0
#pragma unroll
      for (int nb = 0; nb < 8; ++nb)
#pragma unroll
        for (int e = 0; e < 2; ++e)
          cs[nb][e] += mass_ex2(C[blk][nb][2 * hf + e] * c - st[blk][hf].x) * st[blk][hf].y;
#pragma unroll
  for (int nb = 0; nb < 8; ++nb)
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) cs[nb][e] += __shfl_xor_sync(0xffffffffu, cs[nb][e], o);
  if (g == 0) {
#pragma unroll
    for (int nb = 0; nb < 8; ++nb)
#pragma unroll
      for (int e = 0; e < 2; ++e) red[warp * kMassKeys + 8 * nb + 2 * t + e] = cs[nb][e];
  }
  __syncthreads();
  if (threadIdx.x < kMassKeys && kt + (int)threadIdx.x < P) {
    float S = 0.f;
#pragma unroll
    for (int w = 0; w < kMassThreads / 32; ++w) S += red[w * kMassKeys + threadIdx.x];
    colsum[bg * pmax + kt + threadIdx.x] = S;
  }
  __syncthreads();  // buffer `it & 1` and the sums are consumed before they are reused
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
  float2* stats;   // [bh][groups][256]
  float* colsum;   // [bh][groups][P]
};

MassWs carve_mass(const hyq_config* c, int32_t L, void* ws) {
  const size_t bh = (size_t)c->batch * c->num_kv_heads;
  const size_t ng = (size_t)mass_groups(c, c->period);
  char* p = static_cast<char*>(ws) + hyq_select_ws_bytes(c, L);
  MassWs w;
  w.part = reinterpret_cast<float2*>(p);
  p += round_up(bh * ng * kMassSplits * kMassGroupRows * sizeof(float2));
  w.stats = reinterpret_cast<float2*>(p);
  p += round_up(bh * ng * kMassGroupRows * sizeof(float2));
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
         round_up(bh * ng * kMassGroupRows * sizeof(float2)) + round_up(bh * ng * (size_t)(P > 0 ? P : 1) * 4);
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

cudaError_t hyq_launch_select_mass(const hyq_config* c, const void* q_proxy, int32_t n_proxy,
                                   int32_t n_proxy_ld, const void* k_src, int32_t ld, int32_t L,
                                   int32_t* idx_out, int32_t k, void* ws, cudaStream_t s) {
  SelectWs w = carve(c, L, ws);
  MassWs mw = carve_mass(c, L, ws);
  const int32_t P = L - c->window;  // > 0 since k > 0
  const int32_t gq = c->num_q_heads / c->num_kv_heads, R = gq * n_proxy, ng = mass_groups(c, n_proxy);
  const float cs = (float)(1.0 / std::sqrt((double)HYQ_D) / std::log(2.0));  // fl(alpha log2 e)
  const int smem_stats = (kMassGroupRows + 2 * kMassKeys) * kMassStride * 2;  // queries + two key buffers
  const int smem_col = smem_stats + (kMassThreads / 32) * kMassKeys * 4;
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t ea = hyq_once_per_device(attr_done, [&] {
    cudaError_t e = cudaFuncSetAttribute(mass_stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_stats);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(mass_colsum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_col);
    return e;
  });
  if (ea != cudaSuccess) return ea;
  const int n_sm = hyq_num_sms();
  // one block per SM for pass 1 (one fits an SM) and two per SM for pass 2
  const int units = c->num_kv_heads * ng * c->batch;
  const int ns = std::min(kMassSplits, std::max(1, (n_sm + units - 1) / units));
  const int ntiles = (P + kMassKeys - 1) / kMassKeys;
  const int ncol = std::min(ntiles, std::max(1, (2 * n_sm + units - 1) / units));
  const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(q_proxy);
  const __nv_bfloat16* kk = static_cast<const __nv_bfloat16*>(k_src);
  mass_stats_kernel<<<dim3(ns, c->num_kv_heads * ng, c->batch), kMassThreads, smem_stats, s>>>(
      qp, n_proxy, n_proxy_ld, gq, kk, ld, L, cs, R, ng, mw.part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mass_merge_kernel<<<dim3(c->num_kv_heads * ng, c->batch), kMassGroupRows, 0, s>>>(mw.part, mw.stats, R, ng,
                                                                                    ns);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mass_colsum_kernel<<<dim3(ncol, c->num_kv_heads * ng, c->batch), kMassThreads, smem_col, s>>>(qp, n_proxy, n_proxy_ld, gq, kk, ld, P, cs, R, ng, mw.stats, mw.colsum, P);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mass_keys_kernel<<<dim3((P + 255) / 256, c->num_kv_heads, c->batch), 256, 0, s>>>(mw.colsum, ng, P, P, w.keys,
                                                                                   w.err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
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
