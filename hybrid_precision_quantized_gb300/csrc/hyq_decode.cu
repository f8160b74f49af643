// Hybrid-precision decode attention ("HyQuant: Hybrid-Precision Quantization
// for LLM Attention", §4.3 Eq. 8-9 and Appendix A.3 Algorithm 3) and the
// per-step bookkeeping (append to the BF16 tail, proxy-query ring of §5.5).
//
// Work decomposition (one launch, grid S x HKV x B, 16 warps per block):
//   the 4-bit stream of a (batch, KV head) is split along the sequence into
//   S chunks (Algorithm 3, segment 1), and so are its BF16 rows (vertical-
//   line rows, then the tail).  Inside a block every warp works alone on
//   16-row tiles: its 4-bit tiles streamed through its own ring of bulk
//   copies (TMA, no block-wide barrier in the main loop), then its BF16
//   tiles.  Each
//   warp keeps one online-softmax state (m, l, acc) for the g query heads of
//   the KV group, packed into one tensor-core tile (Algorithm 3, "pack g GQA
//   heads").  The block merges its warps; the S block partials are merged by
//   log-sum-exp rescaling (ReduceSoftmax) either inside a thread-block
//   cluster through distributed shared memory, or through the workspace by
//   the last block to finish (an atomic ticket; nobody waits).
//
// 4-bit tiles are dequantised inside the dot products:
//   q.k~  = sum_q s_q (q_q . c_q) + z_q sum(q_q)     (per group q of 32)
//   p v~  = sum_j (p_j s_jq) c_jd + p_j z_jq
// on fp16 mma.sync m16n8k16 with the codes as fp16 subnormals (c * 2^-24,
// one AND per register pair: no offset to cancel, so the fp16 rounding of the
// other operand is not amplified), against the query scaled by an exact power
// of two into fp16 (QK) and against p * s in fp16 (PV); scales, zeros and the
// per-group query sums are applied in fp32.  BF16 tiles are staged by bulk
// copies (or loaded straight into fragment registers); the head_dim order of
// the K products and of the V outputs is permuted (identically in both paths,
// see hyq.h) so that those loads are 16- and 8-byte vectors.  The code
// widths are template parameters: 4- or 8-bit keys (BK) and values (BV), in
// the tile layouts of hyq.h.
#include <cooperative_groups.h>
#include <math.h>

#include "hyq_common.cuh"

namespace cg = cooperative_groups;

namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxSlots = 3;
// BF16 tiles staged in shared memory by a few contiguous bulk copies (K rows,
// then V rows, 256 bytes each): a handful of copies instead of one per row.
constexpr int kFKStride = 256, kFVStride = 256;
constexpr int kFTileBytes = 16 * kFKStride + 16 * kFVStride;  // 8192
constexpr int kFStaged = 7;                                     // staged BF16 tiles per block

// Shared-memory plan for B_K-bit keys and B_V-bit values: each warp streams
// its quantised tiles through a ring of kSlots tiles (3 of 2560 bytes for
// 4-bit codes: 120 KiB of rings; 2 of the larger 8-bit tiles), followed by
// the staged BF16 tiles.
template <int BK, int BV>
struct Dec : QFmt<BK, BV> {
  static constexpr int kSlots = (BK == 4 && BV == 4) ? 3 : 2;
  static constexpr int kRingBytes = kWarps * kSlots * QFmt<BK, BV>::kTile;
  static constexpr int kSmemBytes = kRingBytes + kFStaged * kFTileBytes;
  static_assert(kSlots <= kMaxSlots, "ring barriers");
};
constexpr int kPart = 2 + HYQ_D;                              // m, l, acc[128] per head
constexpr int kMaxSplits = 1024;
// log2(e) / sqrt(128): logits are kept in the base-2 domain.
constexpr float kScale = 0.1275174307366466f;
constexpr float kSubScale = 1.0f / HYQ_F16_SUB_SCALE;         // 2^-24

size_t round_up(size_t x) { return (x + 255) / 256 * 256; }

// Merge modes of the split partials of one (batch, KV head):
//   kDirect  S = 1: the block writes the output itself;
//   kCluster the S blocks form a thread-block cluster and merge through
//            distributed shared memory (no global traffic, no last-block tail);
//   kGlobal  partials go to the workspace and the last block to finish (an
//            atomic ticket; nobody waits) merges them.
enum MergeMode { kDirect = 0, kCluster = 1, kGlobal = 2 };

struct DecodePlan {
  int S;     // blocks per (batch, KV head)
  int mode;  // MergeMode
};

// About one block per SM over all (batch, KV head) pairs, and not more
// blocks than there are 16-row tiles to share; one block per pair when even
// two would not fit in one wave.
// Process-wide settings, written by the two setters from any host thread: the
// plan override packs (merge << 16) | splits into one word so that a launch
// never sees the merge mode of one call with the split count of another.
std::atomic<int32_t> g_plan{0};     // hyq_set_decode_plan override (merge 0 = automatic)
std::atomic<int32_t> g_overlap{0};  // hyq_set_decode_overlap

// overlap: launched as a programmatic dependent, when one SM per merging
// block of the preceding call (assumed of the same shape) is left free, so
// that every block of this call can start while those blocks finish.
DecodePlan decode_plan(const hyq_config* c, int32_t len, bool overlap) {
  const int bh = c->batch * c->num_kv_heads;
  const int sms = hyq_num_sms() - (overlap && 3 * bh <= hyq_num_sms() ? bh : 0);
  int32_t P = len - c->window > 0 ? len - c->window : 0;
  int64_t tiles = (int64_t)(P + 15) / 16 + (hyq_vl_count(c, P) + hyq_cap_tail(c) + 15) / 16;
  // At least ~12 tiles per block: at short contexts fewer, fuller blocks beat
  // one block per SM (Llama-shaped, B1: 1K best at 6 splits, 2K at 12, 4K and
  // longer at the one-wave maximum).
  int cap = (int)(tiles / 12 > 0 ? tiles / 12 : 1);
  DecodePlan p;
  const int32_t plan = g_plan.load(std::memory_order_relaxed);
  if (plan >> 16 != 0) {
    p.mode = (plan >> 16) - 1;
    p.S = p.mode == kDirect ? 1 : plan & 0xFFFF;
    return p;
  }
  if (2 * bh > sms || cap < 2) {  // even two blocks per pair would not fit in one wave
    p.S = 1;
    p.mode = kDirect;
    return p;
  }
  // Measured on GB300 (152 SMs, 8 KV heads, 32K context): the workspace merge
  // at one block per SM beats 16-block clusters, which cannot all be resident
  // with a 185 KiB block each.  S is rounded down: with one block per SM a
  // grid past one wave leaves the last blocks to run after the others (32
  // pairs at S = 5: 160 blocks, 84 us per 32K call against 58 us at S = 4).
  int S = sms / bh;
  if (S > cap) S = cap;
  if (S < 2) S = 2;
  p.S = S;
  p.mode = kGlobal;
  return p;
}

// One decode step's append, fused into the attention launch (hyq_decode_step);
// k_new == nullptr for attention only.
struct StepArgs {
  const __nv_bfloat16* k_new;  // [B][HKV][128]
  const __nv_bfloat16* v_new;
  __nv_bfloat16* k_src;        // [B][HKV][ld][128] or nullptr
  __nv_bfloat16* v_src;
  int32_t ld, period;
  int32_t* tickets_b;          // [B] per-sequence ticket of the counter update
  int32_t overlap;             // launched as a programmatic dependent (hyq_set_decode_overlap)
  // Layout of the next decode call (hyq_decode_step_prefetch), or nullptr:
  // once the block's last warp has read its tiles of this layer, that warp
  // asks L2 to prefetch the share of that layout the same block index will read.
  const uint8_t* nx_qblocks;
  const int32_t* nx_counts;
  const __nv_bfloat16 *nx_vl_k, *nx_vl_v, *nx_tail_k, *nx_tail_v;
};

// floor(i * n / S) for 0 <= i <= S: 32-bit unsigned arithmetic when the
// product fits (the usual case: a few thousand tiles, S <= 1024), else 64-bit.
__device__ __forceinline__ int share_bound(int i, int n, int S) {
  const uint32_t a = (uint32_t)i, nn = (uint32_t)n, s = (uint32_t)S;
  if ((uint64_t)s * nn <= 0xFFFFFFFFull) return (int)(a * nn / s);
  return (int)((uint64_t)a * nn / s);
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}

// The next layout's counts for sequence b, loaded at kernel entry and used
// once they have arrived; clamped to the capacities so that every prefetched
// address lies in that layout's buffers.
struct NextCounts {
  int32_t nq, nvl, ntail;
};
__device__ __forceinline__ NextCounts load_next_counts(const StepArgs& sa, int b) {
  const int32_t* cn = sa.nx_counts + (size_t)b * HYQ_COUNTS;
  return NextCounts{cn[HYQ_CNT_NQ], cn[HYQ_CNT_NVL], cn[HYQ_CNT_NTAIL]};
}
__device__ __forceinline__ NextCounts clamp_next_counts(const NextCounts& n, int nblk_cap, int cap_vl,
                                                        int cap_tail) {
  return NextCounts{min(max(n.nq, 0), nblk_cap * HYQ_QBLOCK_ROWS), min(max(n.nvl, 0), cap_vl),
                    min(max(n.ntail, 0), cap_tail)};
}

// One warp: prefetch into L2 the next layout's quantised tiles [t0, t1) of KV head bh, the share of
// block `split` under the same partition (contiguous, 64 KB per lane).
template <int kTileBytes>
__device__ void prefetch_next_tiles(const StepArgs& sa, const NextCounts& n, size_t bh, int split, int S,
                                    int nblk_cap, int lane) {
  const int nt = (n.nq + 15) >> 4;
  const int t0 = share_bound(split, nt, S), t1 = share_bound(split + 1, nt, S);
  const uint8_t* tiles = sa.nx_qblocks + bh * (size_t)nblk_cap * (4 * kTileBytes) + (size_t)t0 * kTileBytes;
  const uint32_t bytes = (uint32_t)(t1 - t0) * kTileBytes;
  constexpr uint32_t kChunk = 65536;
  for (uint32_t off = lane * kChunk; off < bytes; off += 32 * kChunk)
    prefetch_l2(tiles + off, min(kChunk, bytes - off));
}

// One warp: prefetch into L2 the next layout's BF16 rows [16 f0, 16 f1)
// (vertical lines, then tail) of KV head bh, the share of block `split`.
__device__ void prefetch_next_rows(const StepArgs& sa, const NextCounts& n, size_t bh, int split, int S,
                                   int cap_vl, int cap_tail, int lane) {
  const int32_t nvl = n.nvl, ntail = n.ntail;
  const int nft = (nvl + ntail + 15) >> 4;
  if (lane < 4) {
    const int f0 = share_bound(split, nft, S), f1 = share_bound(split + 1, nft, S);
    const int r0 = 16 * f0, r1 = min(16 * f1, nvl + ntail);
    const bool vpart = lane & 1;
    if (lane < 2 && min(r1, nvl) > r0) {  // vertical-line rows
      const __nv_bfloat16* base = (vpart ? sa.nx_vl_v : sa.nx_vl_k) + (bh * cap_vl + r0) * HYQ_D;
      prefetch_l2(base, (uint32_t)(min(r1, nvl) - r0) * HYQ_D * 2);
    } else if (lane >= 2 && r1 > max(r0, nvl)) {  // tail rows
      const int a = max(r0, nvl) - nvl;
      const __nv_bfloat16* base = (vpart ? sa.nx_tail_v : sa.nx_tail_k) + (bh * cap_tail + a) * HYQ_D;
      prefetch_l2(base, (uint32_t)(r1 - nvl - a) * HYQ_D * 2);
    }
  }
}

// The fused step's counter update: one ticket per (sequence, KV head), taken
// by the block that finishes that pair; the last of the sequence's KV heads
// advances the counters (every block read them at its start, before its own
// pair's ticket).  The increment is a release, so the issuing thread does not
// wait for it; the result is used (with an acquire fence) only at the end.
__device__ __forceinline__ int step_ticket_issue(const StepArgs& sa, int b) {
  int old;
  asm volatile("atom.release.gpu.global.add.s32 %0, [%1], 1;\n" : "=r"(old) : "l"(sa.tickets_b + b) : "memory");
  return old;
}

__device__ __forceinline__ void step_ticket_finish(int old, const StepArgs& sa, const hyq_layout& lay, int b,
                                                   int HKV, bool app, int ntail, int len, int rpos, int rn) {
  if (old != HKV - 1) return;
  asm volatile("fence.acq_rel.gpu;\n" ::: "memory");
  if (app) {
    int32_t* wc = lay.counts + (size_t)b * HYQ_COUNTS;
    wc[HYQ_CNT_NTAIL] = ntail + 1;
    wc[HYQ_CNT_LEN] = len + 1;
    wc[HYQ_CNT_RING_POS] = (rpos + 1) % sa.period;
    wc[HYQ_CNT_RING_N] = min(rn + 1, sa.period);
  }
  sa.tickets_b[b] = 0;
}

// Online-softmax state of one warp for the two heads (2t, 2t+1) a thread owns.
// Logits live in a scaled base-2 domain, lambda' = 2^sigma log2(e) q.k / sqrt(d)
// with one sigma per query head (QConst), chosen so that the per-group query
// sums fit the fp16 operand of the zero-point product; p = 2^((lambda' - m) 2^-sigma).
struct State {
  float m[2];       // running maximum (scaled domain)
  float nm[2];      // -m 2^-sigma (0 while m = -inf)
  float l[2];       // running sum of this thread's probabilities
  float acc[8][4];  // PV accumulators in units of 2^-24
  float zd[4];      // sum_j p_j z_jq: rows g < 4 = group g, columns heads 2t, 2t+1
};

// 2^x on the special-function unit, one instruction (relative error about
// 2^-22; 2^-inf = 0, results below 2^-126 flush to 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Online-softmax update of the two heads (2t, 2t+1) this thread owns with the
// logits of tokens (g, g+8); returns the probabilities p[2r + j].  The
// accumulators are rescaled only when some head's running max moved (the
// factor is exactly 1 otherwise).
// kLazy: first test (one warp vote) whether any logit of the tile exceeds its
// head's running maximum; if none does, the maximum stays, the correction is
// 1 and no cross-lane maximum is needed (the full path would give the same
// bits).  It pays off on long per-warp runs of tiles (one block per
// sequence and KV head), not on short ones, where early tiles move the maximum.
template <bool kLazy>
__device__ __forceinline__ void softmax_update(const float (&lg)[4], State& st, float (&p)[4],
                                               const float (&inv)[2]) {
  if (kLazy) {
    bool above = false;
#pragma unroll
    for (int j = 0; j < 2; ++j) above |= fmaxf(lg[j], lg[2 + j]) > st.m[j];
    if (!__any_sync(0xffffffffu, above)) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        p[j] = ex2(fmaf(lg[j], inv[j], st.nm[j]));
        p[2 + j] = ex2(fmaf(lg[2 + j], inv[j], st.nm[j]));
        st.l[j] += p[j] + p[2 + j];
      }
      return;
    }
  }
  float corr[2];
  bool moved = false;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float tm = fmaxf(lg[j], lg[2 + j]);
    tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 4));
    tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 8));
    tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 16));
    const float mn = fmaxf(st.m[j], tm);
    const float nm = (mn == -INFINITY) ? 0.f : -mn * inv[j];
    moved |= mn != st.m[j];
    corr[j] = ex2(fmaf(st.m[j], inv[j], nm));
    p[j] = ex2(fmaf(lg[j], inv[j], nm));
    p[2 + j] = ex2(fmaf(lg[2 + j], inv[j], nm));
    st.l[j] = fmaf(st.l[j], corr[j], p[j] + p[2 + j]);
    st.m[j] = mn;
    st.nm[j] = nm;
  }
  if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        st.acc[mt][j] *= corr[j];
        st.acc[mt][2 + j] *= corr[j];
      }
      st.zd[j] *= corr[j];
    }
  }
}

// Binary exponent e of a finite x > 0 with x = f 2^e, f in [0.5, 1)
// (subnormals included), 2^k for k in [-126, 127], and the clamp to that range.
__device__ __forceinline__ int exp_of(float x) {
  const int b = __float_as_int(x) >> 23;
  return b != 0 ? b - 126 : (__float_as_int(x * 16777216.f) >> 23) - 150;
}
__device__ __forceinline__ int clamp_exp(int k) { return min(max(k, -126), 127); }
__device__ __forceinline__ float pow2i(int k) { return __int_as_float((clamp_exp(k) + 127) << 23); }
__device__ __forceinline__ bool pos_finite(float x) { return x > 0.f && x <= 3.402823466e38f; }

// Per-block constants of the quantised path.
struct QConst {
  float ksc[2][2];  // scaled-domain factor of the code products [token g (x1) | g+8 (x16 codes)][head 2t + j]
  float inv[2];     // 2^-sigma of heads 2t, 2t+1
  float kss[2];     // scaled-domain factor of the BF16 products 2^sigma log2(e) / sqrt(d), heads 2t, 2t+1
  // B fragment of the zero-point product for head g: the scaled query sums
  // 2^sigma log2(e)/sqrt(d) sum(q over group) of groups 2(t&1), 2(t&1)+1 as
  // an fp16 pair, their high parts for t < 2 and the remainders for t >= 2
  // (hi + lo carries 22 bits).
  uint32_t bz;
};

// The two codes of bytes 1 and 3 of w as the low bytes of two 16-bit halves.
__device__ __forceinline__ uint32_t odd_bytes(uint32_t w) { return __byte_perm(w, 0u, 0x4341); }

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// `n` 32-bit words of a code region: word u of this lane at
// 512 (u / 4) + 16 lane + 4 (u % 4).
template <int n>
__device__ __forceinline__ void load_words(const uint8_t* region, int lane, uint32_t (&w)[n]) {
#pragma unroll
  for (int i = 0; i < n / 4; ++i) {
    const uint4 v = *reinterpret_cast<const uint4*>(region + 512 * i + 16 * lane);
    w[4 * i] = v.x;
    w[4 * i + 1] = v.y;
    w[4 * i + 2] = v.z;
    w[4 * i + 3] = v.w;
  }
}

__device__ __forceinline__ uint32_t u4c(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// One 16-row quantised tile at `tb` (byte layout QFmt<BK, BV>), `vr` valid
// rows.  The codes enter the fp16 MMAs as subnormals c * 2^-24.  4-bit: the
// low nibble of a byte as c * 2^-24, the high nibble, masked in place, as
// 16 c * 2^-24; in both code orders the high nibbles are exactly fragment
// rows g+8 (K: tokens g+8; V: output rows g+8), so the factor 16 is a
// per-row constant: folded into ksc[1] for K and into the epilogue for V.
// 8-bit: bytes 0 and 2 of a word by one AND, bytes 1 and 3 by one byte
// permute, each a fragment register of two codes.  bq holds the query as
// fp16, scaled by 2^e.
//   logit = sum_q s_q (q.c)_q  (per-group code products scaled in fp32)
//         + sum_q z_q (sum q)_q (one MMA: the zero pairs against qc.bz)
//   out  += sum_j (p_j s_jq) c_jd  (P^T scaled by the V scale pairs in fp16)
//         + sum_j p_j z_jq          (one MMA: the V zero pairs against P^T)
template <int BK, int BV, bool kLazy>
__device__ __forceinline__ void q_tile(const uint8_t* tb, int lane, int vr, const uint32_t (&bq)[8][2],
                                       const QConst& qc, State& st) {
  using F = QFmt<BK, BV>;
  const int g = lane >> 2, t = lane & 3;
  float C[4][4];
#pragma unroll
  for (int q = 0; q < 4; ++q) C[q][0] = C[q][1] = C[q][2] = C[q][3] = 0.f;
  if (BK == 4) {
    uint32_t kw[8];
    load_words<8>(tb, lane, kw);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t w = kw[ks], w8 = w >> 8;
      mma_f16(C[ks >> 1], w & 0x000F000Fu, w & 0x00F000F0u, w8 & 0x000F000Fu, w8 & 0x00F000F0u, bq[ks][0],
              bq[ks][1]);
    }
  } else {
    uint32_t kw[16];  // k-step ks: word 2ks (token g), 2ks + 1 (token g + 8)
    load_words<16>(tb, lane, kw);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t w0 = kw[2 * ks], w1 = kw[2 * ks + 1];
      mma_f16(C[ks >> 1], w0 & 0x00FF00FFu, w1 & 0x00FF00FFu, odd_bytes(w0), odd_bytes(w1), bq[ks][0], bq[ks][1]);
    }
  }
  // K metadata of tokens g and g+8: four scales, then four zeros.
  const uint4 ma = *reinterpret_cast<const uint4*>(tb + F::kKMeta + 16 * g);
  const uint4 mb = *reinterpret_cast<const uint4*>(tb + F::kKMeta + 16 * (g + 8));
  const float2 a01 = half2_to_float2(ma.x), a23 = half2_to_float2(ma.y);
  const float2 b01 = half2_to_float2(mb.x), b23 = half2_to_float2(mb.y);
  float lg[4];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    lg[c] = qc.ksc[0][c] * fmaf(a01.x, C[0][c], fmaf(a01.y, C[1][c], fmaf(a23.x, C[2][c], a23.y * C[3][c])));
    lg[2 + c] = qc.ksc[1][c] *
                fmaf(b01.x, C[0][2 + c], fmaf(b01.y, C[1][2 + c], fmaf(b23.x, C[2][2 + c], b23.y * C[3][2 + c])));
  }
  // + sum_q z_q (scaled query sum)_q: the A fragment's k slots 2t, 2t+1 are
  // groups 2(t&1), 2(t&1)+1 (high parts of the sums for t < 2, remainders
  // for t >= 2), so a lane passes the zero pair of those groups.
  mma_f16(lg, (t & 1) ? ma.w : ma.z, (t & 1) ? mb.w : mb.z, 0u, 0u, qc.bz, 0u);
  // A vertical-line position (held in BF16 elsewhere) has NaN key steps in
  // the stream: its logit is NaN, and the row is left out.
#pragma unroll
  for (int i = 0; i < 4; ++i) lg[i] = lg[i] != lg[i] ? -INFINITY : lg[i];
  if (vr < 16) {
    if (g >= vr) lg[0] = lg[1] = -INFINITY;
    if (g + 8 >= vr) lg[2] = lg[3] = -INFINITY;
  }
  float p[4];
  softmax_update<kLazy>(lg, st, p, qc.inv);
  // P^T fragments in fp16: tokens (2t, 2t+1) and (2t+8, 2t+9) of head g.
  const uint32_t pt0 = movmatrix_trans(pack_f16x2(p[0], p[1]));
  const uint32_t pt1 = movmatrix_trans(pack_f16x2(p[2], p[3]));
  const uint8_t* vm = tb + F::kVMeta;
  // V scale pairs of tokens (2t, 2t+1) and (2t+8, 2t+9), groups 0..3.
  const uint4 sv0 = *reinterpret_cast<const uint4*>(vm + 16 * t);
  const uint4 sv1 = *reinterpret_cast<const uint4*>(vm + 16 * (t + 4));
  // sum_j p_j z_jq on the tensor core: A rows = groups (g < 4), k = tokens.
  uint32_t z0 = 0u, z1 = 0u;
  if (g < 4) {
    z0 = *reinterpret_cast<const uint32_t*>(vm + 128 + 16 * t + 4 * g);
    z1 = *reinterpret_cast<const uint32_t*>(vm + 128 + 16 * (t + 4) + 4 * g);
  }
  mma_f16(st.zd, z0, 0u, z1, 0u, pt0, pt1);
  uint32_t vw[BV == 4 ? 8 : 16];
  load_words<BV == 4 ? 8 : 16>(tb + F::kVCode, lane, vw);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    // B operand (tokens x heads) of group q: p * s in packed fp16.
    const uint32_t b0 = hmul2_u32(pt0, u4c(sv0, q)), b1 = hmul2_u32(pt1, u4c(sv1, q));
#pragma unroll
    for (int mm = 0; mm < 2; ++mm) {  // m-tile 2q + mm lies in group q
      if (BV == 4) {
        const uint32_t x = vw[2 * q + mm], x8 = x >> 8;
        mma_f16(st.acc[2 * q + mm], x & 0x000F000Fu, x & 0x00F000F0u, x8 & 0x000F000Fu, x8 & 0x00F000F0u, b0, b1);
      } else {  // m-tile mt: words 2mt (fragment rows g) and 2mt + 1 (rows g + 8)
        const uint32_t y0 = vw[2 * (2 * q + mm)], y1 = vw[2 * (2 * q + mm) + 1];
        mma_f16(st.acc[2 * q + mm], y0 & 0x00FF00FFu, y1 & 0x00FF00FFu, odd_bytes(y0), odd_bytes(y1), b0, b1);
      }
    }
  }
}

// 16 x a bf16 pair (exact: a power of two); the identity for 8-bit values,
// whose accumulator rows carry no factor.
template <int BV>
__device__ __forceinline__ uint32_t row_factor_bf16x2(uint32_t x) {
  if (BV == 8) return x;
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&x);
  v = __hmul2(v, __floats2bfloat162_rn(16.f, 16.f));
  return *reinterpret_cast<uint32_t*>(&v);
}


// One 16-row tile of BF16 rows (rows row0.. of the vertical-line rows followed
// by the tail), `vr` valid rows, loaded directly into fragment registers; row
// `rnew` (a fused step's new row) is read from knew/vnew.  BV: the value code
// width of the quantised tiles, whose accumulator convention the tile follows.
template <int BV, bool kLazy>
__device__ __forceinline__ void f_tile(const __nv_bfloat16* vlk, const __nv_bfloat16* vlv,
                                       const __nv_bfloat16* tk, const __nv_bfloat16* tv, int nvl,
                                       int rnew, const __nv_bfloat16* knew, const __nv_bfloat16* vnew,
                                       int row0, int vr, int lane, const __nv_bfloat16* q_s, const QConst& qc,
                                       State& st) {
  const int g = lane >> 2, t = lane & 3;

  float S[4] = {0.f, 0.f, 0.f, 0.f};
  {
    // K rows g and g+8, chunks t + 4j: the permuted k order of the A fragments.
    uint4 ka[2][4];
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const int rr = g + 8 * a, row = row0 + rr;
      const __nv_bfloat16* src =
          row == rnew ? knew : row < nvl ? vlk + (size_t)row * HYQ_D : tk + (size_t)(row - nvl) * HYQ_D;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        ka[a][j] = rr < vr ? __ldg(reinterpret_cast<const uint4*>(src + 8 * (t + 4 * j))) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int j = ks >> 1, sub = ks & 1;
      const __nv_bfloat16* qe = q_s + g * HYQ_D + 8 * (t + 4 * j) + 4 * sub;  // permuted k order
      mma_bf16(S, u4c(ka[0][j], 2 * sub), u4c(ka[1][j], 2 * sub), u4c(ka[0][j], 2 * sub + 1),
               u4c(ka[1][j], 2 * sub + 1), *reinterpret_cast<const uint32_t*>(qe),
               *reinterpret_cast<const uint32_t*>(qe + 2));
    }
  }
  float lg[4];
  lg[0] = g < vr ? S[0] * qc.kss[0] : -INFINITY;
  lg[1] = g < vr ? S[1] * qc.kss[1] : -INFINITY;
  lg[2] = g + 8 < vr ? S[2] * qc.kss[0] : -INFINITY;
  lg[3] = g + 8 < vr ? S[3] * qc.kss[1] : -INFINITY;
  float p[4];
  softmax_update<kLazy>(lg, st, p, qc.inv);
  // P^T (tokens x heads), scaled by 2^-24 like the 4-bit accumulators.
  const uint32_t b0 = movmatrix_trans(pack_bf16x2(p[0] * kSubScale, p[1] * kSubScale));
  const uint32_t b1 = movmatrix_trans(pack_bf16x2(p[2] * kSubScale, p[3] * kSubScale));
  // V rows 2t + 8b + c, elements 32G + 4g .. +3 for the four groups G.
  uint2 va[4][4];
#pragma unroll
  for (int tk4 = 0; tk4 < 4; ++tk4) {
    const int rr = 2 * t + 8 * (tk4 >> 1) + (tk4 & 1), row = row0 + rr;
    const __nv_bfloat16* src =
        row == rnew ? vnew : row < nvl ? vlv + (size_t)row * HYQ_D : tv + (size_t)(row - nvl) * HYQ_D;
#pragma unroll
    for (int G = 0; G < 4; ++G)
      va[tk4][G] = rr < vr ? __ldg(reinterpret_cast<const uint2*>(src + 32 * G + 4 * g)) : make_uint2(0, 0);
  }
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int G = u >> 1, s2 = u & 1;
    const uint32_t w0 = s2 ? va[0][G].y : va[0][G].x, w1 = s2 ? va[1][G].y : va[1][G].x;
    const uint32_t w2 = s2 ? va[2][G].y : va[2][G].x, w3 = s2 ? va[3][G].y : va[3][G].x;
    // rows g+8 carry the same factor 16 as the 4-bit high-nibble rows
    mma_bf16(st.acc[u], __byte_perm(w0, w1, 0x5410), row_factor_bf16x2<BV>(__byte_perm(w0, w1, 0x7632)),
             __byte_perm(w2, w3, 0x5410), row_factor_bf16x2<BV>(__byte_perm(w2, w3, 0x7632)), b0, b1);
  }
}

// The same BF16 tile from shared memory (K rows at stride kFKStride, V rows
// at kFVStride); rows at or past `vr` are masked (their contents are undefined).
// The unpadded rows cost 2-way (K) and 4-way (V) bank conflicts on these few
// loads, against 32 single-row copies per tile otherwise.
template <int BV, bool kLazy>
__device__ __forceinline__ void f_tile_smem(const uint8_t* Ks, const uint8_t* Vs, int vr, int lane,
                                            const __nv_bfloat16* q_s, const QConst& qc, State& st) {
  const int g = lane >> 2, t = lane & 3;

  float S[4] = {0.f, 0.f, 0.f, 0.f};
  {
    uint4 ka[2][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        ka[a][j] = *reinterpret_cast<const uint4*>(Ks + (g + 8 * a) * kFKStride + 16 * (t + 4 * j));
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int j = ks >> 1, sub = ks & 1;
      const __nv_bfloat16* qe = q_s + g * HYQ_D + 8 * (t + 4 * j) + 4 * sub;  // permuted k order
      mma_bf16(S, u4c(ka[0][j], 2 * sub), u4c(ka[1][j], 2 * sub), u4c(ka[0][j], 2 * sub + 1),
               u4c(ka[1][j], 2 * sub + 1), *reinterpret_cast<const uint32_t*>(qe),
               *reinterpret_cast<const uint32_t*>(qe + 2));
    }
  }
  float lg[4];
  lg[0] = g < vr ? S[0] * qc.kss[0] : -INFINITY;
  lg[1] = g < vr ? S[1] * qc.kss[1] : -INFINITY;
  lg[2] = g + 8 < vr ? S[2] * qc.kss[0] : -INFINITY;
  lg[3] = g + 8 < vr ? S[3] * qc.kss[1] : -INFINITY;
  float p[4];
  softmax_update<kLazy>(lg, st, p, qc.inv);
  const uint32_t b0 = movmatrix_trans(pack_bf16x2(p[0] * kSubScale, p[1] * kSubScale));
  const uint32_t b1 = movmatrix_trans(pack_bf16x2(p[2] * kSubScale, p[3] * kSubScale));
  uint2 va[4][4];
#pragma unroll
  for (int tk4 = 0; tk4 < 4; ++tk4) {
    const int rr = 2 * t + 8 * (tk4 >> 1) + (tk4 & 1);
#pragma unroll
    for (int G = 0; G < 4; ++G)
      va[tk4][G] = rr < vr ? *reinterpret_cast<const uint2*>(Vs + rr * kFVStride + 2 * (32 * G + 4 * g))
                           : make_uint2(0, 0);
  }
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int G = u >> 1, s2 = u & 1;
    const uint32_t w0 = s2 ? va[0][G].y : va[0][G].x, w1 = s2 ? va[1][G].y : va[1][G].x;
    const uint32_t w2 = s2 ? va[2][G].y : va[2][G].x, w3 = s2 ? va[3][G].y : va[3][G].x;
    // rows g+8 carry the same factor 16 as the 4-bit high-nibble rows
    mma_bf16(st.acc[u], __byte_perm(w0, w1, 0x5410), row_factor_bf16x2<BV>(__byte_perm(w0, w1, 0x7632)),
             __byte_perm(w2, w3, 0x5410), row_factor_bf16x2<BV>(__byte_perm(w2, w3, 0x7632)), b0, b1);
  }
}

template <int kMode, int BK, int BV>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(
    const __nv_bfloat16* __restrict__ q, hyq_layout lay, __nv_bfloat16* __restrict__ out,
    int32_t* __restrict__ tickets, float* __restrict__ part, int HQ, int gq, int nblk_cap,
    int cap_vl, int cap_tail, int S, const StepArgs sa) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(16) __nv_bfloat16 q_s[HYQ_MAX_GQA * HYQ_D];
  // B fragments of the query, [k-step pair][row g][lane t][4]: a lane's four
  // 16-byte loads are consecutive across the warp (no bank conflicts).
  __shared__ __align__(16) uint32_t bq_s[4][HYQ_MAX_GQA][4][4];
  __shared__ float rowc_s[HYQ_MAX_GQA][4];                       // per query row: ksc (x1, x16), 2^-sigma, kss
  __shared__ uint32_t bz_s[HYQ_MAX_GQA][4];                      // per query row and lane t: zero-point B fragment
  __shared__ __align__(8) uint64_t bars[kWarps * kMaxSlots];
  __shared__ __align__(8) uint64_t fbars[kFStaged];
  __shared__ __align__(8) uint64_t qbar;
  __shared__ float red_m[kWarps][HYQ_MAX_GQA], red_l[kWarps][HYQ_MAX_GQA];
  __shared__ float sL[HYQ_MAX_GQA];
  __shared__ int s_flag;

  using D = Dec<BK, BV>;
  constexpr int kSlots = D::kSlots, kTile = D::kTile;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z, HKV = gridDim.y;
  const size_t bh = (size_t)b * HKV + h;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;

  // With overlap this launch reads only the cache layout before
  // griddepcontrol.wait (the caller guarantees the preceding kernel does not
  // write it), and the query, the new row and every output after it; it lets
  // the next launch start only once that wait has returned, so that every
  // kernel but the immediately preceding one has finished whenever a launch
  // starts.
  const bool ovl = sa.overlap != 0;
  // The query rows of the KV group: plain 16-byte loads issued first (a
  // load returns well before a bulk copy would), stored to shared memory
  // just before the block barrier below.  With overlap the query may only be
  // read after griddepcontrol.wait and comes by bulk copy there.
  if (tid == 0) {
    mbar_init(&qbar, 1);
    mbar_fence_init();
  }
  const int nq16 = gq * HYQ_D / 8;
  if (ovl && tid == 0) {
    // Warm L2 (and the address translation) for the query rows, which may
    // only be read after griddepcontrol.wait; a prefetch returns no data, so
    // it is correct whatever the preceding kernel still writes there.
    prefetch_l2(q + ((size_t)b * HQ + (size_t)h * gq) * HYQ_D, gq * HYQ_D * 2);
    if (sa.k_new) {
      prefetch_l2(sa.k_new + bh * HYQ_D, HYQ_D * 2);
      prefetch_l2(sa.v_new + bh * HYQ_D, HYQ_D * 2);
    }
  }
  uint4 qv = make_uint4(0, 0, 0, 0);
  if (!ovl && tid < nq16)
    qv = __ldg(reinterpret_cast<const uint4*>(q + ((size_t)b * HQ + (size_t)h * gq) * HYQ_D) + tid);
  const int32_t* cnt = lay.counts + (size_t)b * HYQ_COUNTS;
  int32_t nq = cnt[HYQ_CNT_NQ], nvl = cnt[HYQ_CNT_NVL], ntail = cnt[HYQ_CNT_NTAIL];
  const bool next_cnt_loaded = sa.nx_counts != nullptr;
  NextCounts nxraw{0, 0, 0};
  if (next_cnt_loaded && warp == kWarps - 1) nxraw = load_next_counts(sa, b);
  if (nq < 0 || nq > nblk_cap * HYQ_QBLOCK_ROWS || nvl < 0 || nvl > cap_vl || ntail < 0 || ntail > cap_tail) {
    if (tid == 0 && split == 0) hyq_set_err(lay.err, HYQ_DEVERR_COUNT);
    nq = min(max(nq, 0), nblk_cap * HYQ_QBLOCK_ROWS);
    nvl = min(max(nvl, 0), cap_vl);
    ntail = min(max(ntail, 0), cap_tail);
  }
  // Fused step: this token's K/V row becomes tail row `ntail` (when it fits).
  const bool step = sa.k_new != nullptr;
  int32_t len = 0, rpos = 0, rn = 0;
  bool app = false;
  if (step) {
    len = cnt[HYQ_CNT_LEN];
    rpos = cnt[HYQ_CNT_RING_POS];
    rn = cnt[HYQ_CNT_RING_N];
    app = ntail < cap_tail && len >= 0 && rpos >= 0 && rpos < sa.period && (sa.k_src == nullptr || len < sa.ld);
    if (!app && tid == 0 && split == 0 && h == 0) hyq_set_err(lay.err, HYQ_DEVERR_COUNT);
  }
  // This block's share of the 4-bit tiles and of the BF16 tiles.
  const int nt = (nq + 15) >> 4, nf = nvl + ntail + (app ? 1 : 0), nft = (nf + 15) >> 4;
  const int t0 = share_bound(split, nt, S), t1 = share_bound(split + 1, nt, S);
  const int f0 = share_bound(split, nft, S), f1 = share_bound(split + 1, nft, S);
  // 4-bit tiles go round-robin over the warps, starting after the warps that
  // also take a BF16 tile.
  const int ntc = t1 - t0, rot = (f1 - f0) % kWarps;
  const int my0 = (warp - rot + kWarps) % kWarps;
  const int nj = ntc > my0 ? (ntc - my0 + kWarps - 1) / kWarps : 0;
  const uint8_t* tiles = lay.qblocks + bh * (size_t)nblk_cap * D::kBlock;
  uint8_t* ring = smem + warp * kSlots * kTile;
  uint64_t* wb = bars + warp * kSlots;
  const __nv_bfloat16* vlk = static_cast<const __nv_bfloat16*>(lay.vl_k) + bh * cap_vl * HYQ_D;
  const __nv_bfloat16* vlv = static_cast<const __nv_bfloat16*>(lay.vl_v) + bh * cap_vl * HYQ_D;
  const __nv_bfloat16* tk = static_cast<const __nv_bfloat16*>(lay.tail_k) + bh * cap_tail * HYQ_D;
  const __nv_bfloat16* tv = static_cast<const __nv_bfloat16*>(lay.tail_v) + bh * cap_tail * HYQ_D;
  const int n_staged = min(f1 - f0, kFStaged);
  // Fused step: the block holding the new row stores it (tail, caller's BF16
  // cache) and the group's queries (proxy ring) at its end; nothing in this
  // launch reads those slots.  Warp 2 loads the row now, off the critical path.
  const bool owner = app && (nvl + ntail) >> 4 >= f0 && (nvl + ntail) >> 4 < f1;
  uint4 nrow = make_uint4(0, 0, 0, 0);
  if (owner && warp == 2 && !ovl)
    nrow = __ldg(reinterpret_cast<const uint4*>((lane >= 16 ? sa.v_new : sa.k_new) + bh * HYQ_D) + (lane & 15));
  uint8_t* fstage = smem + D::kRingBytes + warp * kFTileBytes;
  // A warp's ring and staging barriers are its own: lane 0 initialises them
  // and the warp issues its first copies at once, behind the query copy
  // issued at entry, so that the preparation of the query below overlaps
  // their latency.
  if (lane == 0) {
    for (int i = 0; i < kSlots; ++i) mbar_init(&wb[i], 1);
    if (warp < n_staged) mbar_init(&fbars[warp], 1);
    mbar_fence_init();
  }
  __syncwarp();
  // Ring slot i is always filled by lane i: the bulk copies one thread issues
  // complete one after another, so one issuing lane per slot keeps all of a
  // warp's slots in flight at once.
  if (lane < kSlots && lane < nj) {
    const int j = lane;
    mbar_arrive_expect_tx(&wb[j], kTile);
    bulk_g2s(ring + j * kTile, tiles + (size_t)(t0 + my0 + kWarps * j) * kTile, kTile, &wb[j]);
  }
  if (warp < n_staged) {
    // The first kFStaged BF16 tiles of this block: the rows of a tile are
    // contiguous in the vertical-line buffer and in the tail, so a tile takes
    // one K and one V copy per buffer it touches, issued by lanes 4 and 5
    // (not by the ring lanes).  Used after the 4-bit loop.
    const int row0 = 16 * (f0 + warp), nrows = min(16, nf - row0);
    // the new row of a fused step (if in this tile) comes from the input instead
    const int rnew = app ? nvl + ntail - row0 : -1;
    const int ncopy = nrows - ((rnew >= 0 && rnew < nrows) ? 1 : 0);
    const int na = max(0, min(row0 + nrows, nvl) - row0);  // rows in the vertical-line buffer
    const int ntr = min(nrows - na, ntail - max(0, row0 + na - nvl));  // stored tail rows (not the new one)
    if (lane == 4) mbar_arrive_expect_tx(&fbars[warp], ncopy * 2 * HYQ_D * 2);
    __syncwarp();
    if (lane == 4 && na > 0) {
      bulk_g2s(fstage, vlk + (size_t)row0 * HYQ_D, na * HYQ_D * 2, &fbars[warp]);
      bulk_g2s(fstage + 16 * kFKStride, vlv + (size_t)row0 * HYQ_D, na * HYQ_D * 2, &fbars[warp]);
    }
    if (lane == 5 && ntr > 0) {
      const int tr = row0 + na - nvl;  // first tail row
      bulk_g2s(fstage + na * kFKStride, tk + (size_t)tr * HYQ_D, ntr * HYQ_D * 2, &fbars[warp]);
      bulk_g2s(fstage + 16 * kFKStride + na * kFVStride, tv + (size_t)tr * HYQ_D, ntr * HYQ_D * 2, &fbars[warp]);
    }
  }
  for (int i = gq * HYQ_D / 8 + tid; i < HYQ_MAX_GQA * HYQ_D / 8; i += kThreads)
    reinterpret_cast<uint4*>(q_s)[i] = make_uint4(0, 0, 0, 0);  // query rows past g
  if (!ovl && tid < nq16) reinterpret_cast<uint4*>(q_s)[tid] = qv;
  __syncthreads();
  if (ovl) {
    // The layout copies are in flight; now wait for the preceding kernel and
    // fetch what it may have produced.
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    if (tid == 0) {
      mbar_arrive_expect_tx(&qbar, gq * HYQ_D * 2);
      bulk_g2s(q_s, q + ((size_t)b * HQ + (size_t)h * gq) * HYQ_D, gq * HYQ_D * 2, &qbar);
    }
    if (owner && warp == 2)
      nrow = __ldg(reinterpret_cast<const uint4*>((lane >= 16 ? sa.v_new : sa.k_new) + bh * HYQ_D) + (lane & 15));
    if (!mbar_wait(&qbar, 0) && tid == 0) hyq_set_err(lay.err, HYQ_DEVERR_TIMEOUT);
  }
  if (owner && warp == 2) {
    // the new row into its staging slot (the tile's bulk copies skip it); the
    // barrier before the main loop orders this for the warp that reads it
    const int fw = ((nvl + ntail) >> 4) - f0, rin = (nvl + ntail) & 15;
    if (fw < n_staged)
      reinterpret_cast<uint4*>(smem + D::kRingBytes + fw * kFTileBytes + (lane >= 16 ? 16 * kFKStride : 0) +
                               rin * kFKStride)[lane & 15] = nrow;
  }
  // One warp per query row (rows past g stay zero): the row's fp16 B
  // fragments, scaled by an exact power of two 2^qe so that max |q| lies in
  // [2^13, 2^14), stored in the order lane (g, t) reads them; and the row's
  // constants: sigma (its largest scaled group sum 2^sigma log2(e)/sqrt(d)
  // |sum q| below 2^13, and sigma <= 23 - exponent(max |q|), which bounds the
  // scaled logits), the code-product factors and the zero-point fragments.
  if (warp < HYQ_MAX_GQA) {
    const int r = warp;
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (r < gq) {
      const uint2 v = *reinterpret_cast<const uint2*>(q_s + r * HYQ_D + 4 * lane);
      const float2 x01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
      const float2 x23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
      x[0] = x01.x, x[1] = x01.y, x[2] = x23.x, x[3] = x23.y;
    }
    float gs = (x[0] + x[1]) + (x[2] + x[3]);  // group lane / 8
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) gs += __shfl_xor_sync(0xffffffffu, gs, o);
    float am = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
    float gm = fabsf(gs * kScale);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
#pragma unroll
    for (int o = 8; o < 32; o <<= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
    const int qe = pos_finite(am) ? clamp_exp(14 - exp_of(am)) : 14;
    const float gmb = fmaxf(gm, am * 0.0009765625f);  // 2^-10 max |q|
    const int sg = pos_finite(gmb) ? clamp_exp(13 - exp_of(gmb)) : 13;
    const float qscale = pow2i(qe);
#pragma unroll
    for (int hp = 0; hp < 2; ++hp) {
      const int e = 4 * lane + 2 * hp;  // pair (e, e + 1) -> lane t, k-step ks, half hh
      const int hh = (e >> 1) & 1;
      const int tt = BK == 4 ? (e >> 3) & 3 : (e >> 2) & 3;
      const int ks = BK == 4 ? 2 * (e >> 5) + ((e >> 2) & 1) : e >> 4;
      bq_s[ks >> 1][r][tt][2 * (ks & 1) + hh] = pack_f16x2(x[2 * hp] * qscale, x[2 * hp + 1] * qscale);
    }
    const float kss = kScale * pow2i(sg);
    const float s0 = __shfl_sync(0xffffffffu, gs, 0) * kss, s1 = __shfl_sync(0xffffffffu, gs, 8) * kss;
    const float s2 = __shfl_sync(0xffffffffu, gs, 16) * kss, s3 = __shfl_sync(0xffffffffu, gs, 24) * kss;
    if (lane < 4) {  // lane = t of the reading thread
      const float y0 = (lane & 1) ? s2 : s0, y1 = (lane & 1) ? s3 : s1;
      const float h0 = __half2float(__float2half_rn(y0)), h1 = __half2float(__float2half_rn(y1));
      bz_s[r][lane] = lane < 2 ? pack_f16x2(h0, h1) : pack_f16x2(y0 - h0, y1 - h1);
    }
    if (lane == 0) {
      const float k0 = kScale * pow2i(clamp_exp(24 - qe)) * pow2i(sg);
      rowc_s[r][0] = k0;
      rowc_s[r][1] = BK == 4 ? k0 * 0.0625f : k0;  // 4-bit tokens g+8 carry 16 c
      rowc_s[r][2] = pow2i(-sg);
      rowc_s[r][3] = kss;
    }
  }
  __syncthreads();
  // B fragments of q in the permuted k order of the key codes: kstep ks
  // covers elements e + {0,1} and e + {2,3}, e = 8(t + 4(ks/2)) + 4(ks%2)
  // for 4-bit keys, e = 16 ks + 4t for 8-bit keys.
  uint32_t bq[8][2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 v = *reinterpret_cast<const uint4*>(&bq_s[i][g][t][0]);
    bq[2 * i][0] = v.x, bq[2 * i][1] = v.y, bq[2 * i + 1][0] = v.z, bq[2 * i + 1][1] = v.w;
  }
  QConst qc;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    qc.ksc[0][j] = rowc_s[2 * t + j][0];
    qc.ksc[1][j] = rowc_s[2 * t + j][1];
    qc.inv[j] = rowc_s[2 * t + j][2];
    qc.kss[j] = rowc_s[2 * t + j][3];
  }
  qc.bz = bz_s[g][t];

  State st;
  st.m[0] = st.m[1] = -INFINITY;
  st.nm[0] = st.nm[1] = 0.f;
  st.l[0] = st.l[1] = 0.f;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) st.acc[mt][0] = st.acc[mt][1] = st.acc[mt][2] = st.acc[mt][3] = 0.f;
  st.zd[0] = st.zd[1] = st.zd[2] = st.zd[3] = 0.f;

  // Next-layer L2 prefetch (hyq_decode_step_prefetch): issued by the last
  // warp once its own tiles are read (the next layout's counters, loaded at
  // entry, have long arrived), so that it keeps HBM busy through this
  // launch's reductions and merge.  Issued at the warp's first tile instead,
  // it slowed the call (18.96 against 15.95 us at the 32K layer): the
  // prefetch then competes with this layer's own reads.
  const bool pf_warp = next_cnt_loaded && warp == kWarps - 1;
  auto issue_prefetch = [&]() {
    const NextCounts nxc = clamp_next_counts(nxraw, nblk_cap, cap_vl, cap_tail);
    // Only a next layer that fits comfortably in L2 (its estimate from this
    // sequence's counts below half of the 129 MB) is worth prefetching; a
    // larger one would only evict lines before they are used.
    const double next_bytes = (double)gridDim.z * HKV *
                              ((double)((nxc.nq + 15) >> 4) * kTile + (double)(nxc.nvl + nxc.ntail) * 4 * HYQ_D);
    if (next_bytes > 64.0 * 1024 * 1024) return;
    prefetch_next_tiles<kTile>(sa, nxc, bh, split, S, nblk_cap, lane);
    prefetch_next_rows(sa, nxc, bh, split, S, cap_vl, cap_tail, lane);
  };

  // ---- 4-bit tiles through the warp's ring ---------------------------------
  for (int j = 0; j < nj; ++j) {
    const int slot = j % kSlots;
    const bool ok = mbar_wait(&wb[slot], (j / kSlots) & 1);
    if (__any_sync(0xffffffffu, !ok)) {
      // A copy did not arrive: flag it, and make sure none of this warp's
      // copies is still in flight before shared memory is reused below.
      if (lane == 0) {
        hyq_set_err(lay.err, HYQ_DEVERR_TIMEOUT);
        for (int jj = j; jj < nj && jj < j + kSlots; ++jj) (void)mbar_wait(&wb[jj % kSlots], (jj / kSlots) & 1);
      }
      __syncwarp();
      break;
    }
    const int tile = t0 + my0 + kWarps * j;
    q_tile<BK, BV, kMode == kDirect>(ring + slot * kTile, lane, min(16, nq - 16 * tile), bq, qc, st);
    __syncwarp();
    if (lane == slot && j + kSlots < nj) {
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      mbar_arrive_expect_tx(&wb[slot], kTile);
      bulk_g2s(ring + slot * kTile, tiles + (size_t)(tile + kWarps * kSlots) * kTile, kTile, &wb[slot]);
    }
  }

  // ---- BF16 tiles (vertical-line rows, then the tail): the staged ones have
  // long arrived by now -----------------------------------------------------
  if (warp < n_staged) {
    const bool ok = mbar_wait(&fbars[warp], 0);
    if (__any_sync(0xffffffffu, !ok)) {
      if (lane == 0) {
        hyq_set_err(lay.err, HYQ_DEVERR_TIMEOUT);
        (void)mbar_wait(&fbars[warp], 0);
      }
      __syncwarp();
    } else {
      f_tile_smem<BV, kMode == kDirect>(fstage, fstage + 16 * kFKStride, min(16, nf - 16 * (f0 + warp)), lane, q_s,
                                        qc, st);
    }
  }
  for (int fi = f0 + kFStaged + warp; fi < f1; fi += kWarps)  // tiles past the staged ones
    f_tile<BV, kMode == kDirect>(vlk, vlv, tk, tv, nvl, app ? nvl + ntail : -1, sa.k_new + bh * HYQ_D,
                                 sa.v_new + bh * HYQ_D, 16 * fi, min(16, nf - 16 * fi), lane, q_s, qc, st);

  if (pf_warp) issue_prefetch();
  // ---- warp partial -> this warp's own ring (every copy into it has been
  // consumed): acc[head][128] with the zero-point terms, (m, l) per head -----
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) st.l[j] += __shfl_xor_sync(0xffffffffu, st.l[j], o);
  // sum_j p_j z_jq of heads 2t, 2t+1 sits in lane (q, t): gather all four groups.
  float zt[4][2];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    zt[q][0] = __shfl_sync(0xffffffffu, st.zd[0], 4 * q + t);
    zt[q][1] = __shfl_sync(0xffffffffu, st.zd[1], 4 * q + t);
  }
  // [8 heads][128] = 4 KB <= the ring; element d of head hd at hd*128 + (d ^ (hd/2)),
  // so that the 32 lanes' stores of one accumulator fall in 32 banks.
  float* wpart = reinterpret_cast<float*>(ring);
  // Accumulator (m-tile u, ci) of thread (g, t): element 32(u/2) + 4g +
  // 2(u%2) + (ci >> 1), head 2t + (ci & 1); with 4-bit values the rows
  // ci >= 2 carry 16 c.
#pragma unroll
  for (int u = 0; u < 8; ++u)
#pragma unroll
    for (int ci = 0; ci < 4; ++ci) {
      const int d = 32 * (u >> 1) + 4 * g + 2 * (u & 1) + (ci >> 1), hd = 2 * t + (ci & 1);
      const float f = (BV == 4 && ci >= 2) ? HYQ_F16_SUB_SCALE / 16.f : HYQ_F16_SUB_SCALE;
      wpart[hd * HYQ_D + (d ^ t)] = fmaf(st.acc[u][ci], f, zt[u >> 1][ci & 1]);
    }
  if (g == 0)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      red_m[warp][2 * t + j] = st.m[j] == -INFINITY ? -INFINITY : st.m[j] * qc.inv[j];  // back to log2 units
      red_l[warp][2 * t + j] = st.l[j];
    }
  __syncthreads();
  // ---- block partial: thread i takes elements i, i + 512 (a warp shares one
  // head); the warps' weights 2^(m_w - M) come from lanes 0..15 by shuffle --
  float* blk = reinterpret_cast<float*>(smem + D::kRingBytes);  // [head][2 + 128] (staged area, consumed)
  float* pp = part + (bh * S + split) * (size_t)(HYQ_MAX_GQA * kPart);
  for (int i = tid; i < gq * HYQ_D; i += kThreads) {
    const int hd = i >> 7, d = i & (HYQ_D - 1);
    const float mw = lane < kWarps ? red_m[lane][hd] : -INFINITY;
    float M = mw;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float Ms = (M == -INFINITY) ? 0.f : M;
    const float wt = lane < kWarps ? ex2(mw - Ms) : 0.f;
    float Lsum = lane < kWarps ? red_l[lane][hd] * wt : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, o);
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
      a = fmaf(__shfl_sync(0xffffffffu, wt, w),
               reinterpret_cast<const float*>(smem + w * kSlots * kTile)[hd * HYQ_D + (d ^ (hd >> 1))], a);
    if (kMode == kDirect) {
      out[((size_t)b * HQ + (size_t)h * gq + hd) * HYQ_D + d] = __float2bfloat16_rn(Lsum > 0.f ? a / Lsum : 0.f);
    } else {
      float* dst = kMode == kCluster ? blk : pp;
      dst[hd * kPart + 2 + d] = a;
      if (d == 0) {
        dst[hd * kPart + 0] = M;
        dst[hd * kPart + 1] = Lsum;
      }
    }
  }
  if (owner) {
    if (warp == 2) {
      const size_t row = (bh * cap_tail + ntail) * HYQ_D;
      reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(lane >= 16 ? lay.tail_v : lay.tail_k) + row)[lane & 15] = nrow;
      if (sa.k_src)
        reinterpret_cast<uint4*>((lane >= 16 ? sa.v_src : sa.k_src) + (bh * sa.ld + len) * HYQ_D)[lane & 15] = nrow;
    } else if (tid >= 96 && tid < 96 + 16 * gq) {
      const int r = (tid - 96) >> 4, c8 = tid & 15;
      const size_t hq = (size_t)b * HQ + (size_t)h * gq + r;
      reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(lay.q_ring) + (hq * sa.period + rpos) * HYQ_D)[c8] =
          reinterpret_cast<const uint4*>(q_s + r * HYQ_D)[c8];
    }
  }
  const bool ticket_thread = step && tid == kThreads - 1;
  if (kMode == kDirect) {
    if (ticket_thread) step_ticket_finish(step_ticket_issue(sa, b), sa, lay, b, HKV, app, ntail, len, rpos, rn);
    return;
  }

  if (kMode == kCluster) {
    // ---- ReduceSoftmax across the cluster through distributed shared memory
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();  // every block's partial is in its shared memory
    float* rm = reinterpret_cast<float*>(smem);  // [S][8] remote m, then weights (rings are free now)
    float* rl = rm + 16 * HYQ_MAX_GQA;          // [S][8] remote l
    for (int i = tid; i < S * gq; i += kThreads) {
      const int r = i / gq, hd = i % gq;
      const float* rb = cluster.map_shared_rank(blk, r);
      rm[r * HYQ_MAX_GQA + hd] = rb[hd * kPart + 0];
      rl[r * HYQ_MAX_GQA + hd] = rb[hd * kPart + 1];
    }
    __syncthreads();
    if (tid < gq) {
      float M = -INFINITY;
      for (int r = 0; r < S; ++r) M = fmaxf(M, rm[r * HYQ_MAX_GQA + tid]);
      const float Ms = (M == -INFINITY) ? 0.f : M;
      float Lsum = 0.f;
      for (int r = 0; r < S; ++r) {
        const float wt = ex2(rm[r * HYQ_MAX_GQA + tid] - Ms);
        rm[r * HYQ_MAX_GQA + tid] = wt;
        Lsum = fmaf(rl[r * HYQ_MAX_GQA + tid], wt, Lsum);
      }
      sL[tid] = Lsum;
    }
    __syncthreads();
    // Block `split` of the cluster writes its share of the (head, element) outputs.
    const int items = gq * HYQ_D, per = (items + S - 1) / S;
    for (int i = split * per + tid; i < min(items, (split + 1) * per); i += kThreads) {
      const int hd = i >> 7, d = i & (HYQ_D - 1);
      float a = 0.f;
#pragma unroll 4
      for (int r = 0; r < S; ++r) {
        const float* rb = cluster.map_shared_rank(blk, r);
        a = fmaf(rb[hd * kPart + 2 + d], rm[r * HYQ_MAX_GQA + hd], a);
      }
      const float Lh = sL[hd];
      out[((size_t)b * HQ + (size_t)h * gq + hd) * HYQ_D + d] = __float2bfloat16_rn(Lh > 0.f ? a / Lh : 0.f);
    }
    cluster.sync();  // no block leaves while another still reads its shared memory
    if (ticket_thread && split == 0)
      step_ticket_finish(step_ticket_issue(sa, b), sa, lay, b, HKV, app, ntail, len, rpos, rn);
    return;
  }

  // ---- kGlobal: the last block to finish merges the workspace partials -----
  // The barrier orders every thread's partial writes before thread 0's
  // release; its acquire (in the last block) orders them before the reads.
  __syncthreads();
  if (tid == 0) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;\n" : "=r"(old) : "l"(tickets + bh) : "memory");
    s_flag = (old == S - 1);
  }
  __syncthreads();
  if (!s_flag) return;
  const int tk_old = ticket_thread ? step_ticket_issue(sa, b) : 0;  // overlaps the merge
  const float* pb = part + bh * S * (size_t)(HYQ_MAX_GQA * kPart);
  constexpr size_t kSplitStride = HYQ_MAX_GQA * kPart;
  // Thread i merges element i (and i + 512) of head i >> 7 (one head per
  // warp): lanes load the splits' (m, l) of that head, 32 splits at a time,
  // every thread its element of those splits, all in one round trip; the
  // weights reach the other lanes by shuffle.
  for (int i = tid; i < gq * HYQ_D; i += kThreads) {
    const int hd = i >> 7, d = i & (HYQ_D - 1);
    const float* e = pb + hd * kPart + 2 + d;
    float M = -INFINITY;
    if (S > 32)  // a first pass for the maximum over all splits
      for (int s0 = 0; s0 < S; s0 += 32)
        M = fmaxf(M, s0 + lane < S ? __ldcg(pb + (size_t)(s0 + lane) * kSplitStride + hd * kPart) : -INFINITY);
    float a = 0.f, Lsum = 0.f;
    for (int s0 = 0; s0 < S; s0 += 32) {
      const int sl = s0 + lane;
      const float mw = sl < S ? __ldcg(pb + (size_t)sl * kSplitStride + hd * kPart) : -INFINITY;
      const float lw = sl < S ? __ldcg(pb + (size_t)sl * kSplitStride + hd * kPart + 1) : 0.f;
      float v[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] = s0 + k < S ? __ldcg(e + (size_t)(s0 + k) * kSplitStride) : 0.f;
      float Mc = fmaxf(M, mw);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) Mc = fmaxf(Mc, __shfl_xor_sync(0xffffffffu, Mc, o));
      M = Mc;  // S <= 32: the maximum of this (only) chunk; S > 32: the first pass's
      const float Ms = (M == -INFINITY) ? 0.f : M;
      const float wt = sl < S ? ex2(mw - Ms) : 0.f;
      float lsum = lw * wt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
      Lsum += lsum;
#pragma unroll
      for (int k = 0; k < 32; ++k) a = fmaf(__shfl_sync(0xffffffffu, wt, k), v[k], a);
    }
    out[((size_t)b * HQ + (size_t)h * gq + hd) * HYQ_D + d] = __float2bfloat16_rn(Lsum > 0.f ? a / Lsum : 0.f);
  }
  if (tid == 0) tickets[bh] = 0;
  if (ticket_thread) step_ticket_finish(tk_old, sa, lay, b, HKV, app, ntail, len, rpos, rn);
}

// One step's append: BF16 tail row, proxy ring slot, optional BF16 source row.
// grid (B), 256 threads.
__global__ void decode_append_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_new,
                                     const __nv_bfloat16* __restrict__ v_new, hyq_layout lay,
                                     __nv_bfloat16* k_src, __nv_bfloat16* v_src, int32_t ld, int HQ,
                                     int HKV, int period, int cap_tail) {
  __shared__ int s_ok, s_ntail, s_len, s_pos;
  const int b = blockIdx.x, tid = threadIdx.x;
  int32_t* cnt = lay.counts + (size_t)b * HYQ_COUNTS;
  if (tid == 0) {
    s_ntail = cnt[HYQ_CNT_NTAIL];
    s_len = cnt[HYQ_CNT_LEN];
    s_pos = cnt[HYQ_CNT_RING_POS];
    bool ok = s_ntail >= 0 && s_ntail < cap_tail && s_len >= 0 && s_pos >= 0 && s_pos < period &&
              (k_src == nullptr || s_len < ld);
    if (!ok) hyq_set_err(lay.err, HYQ_DEVERR_COUNT);
    s_ok = ok;
  }
  __syncthreads();
  if (!s_ok) return;
  const int ntail = s_ntail, len = s_len, pos = s_pos;
  // q -> ring[b][h][pos]
  for (int i = tid; i < HQ * HYQ_D / 8; i += blockDim.x) {
    const int hq = i >> 4, c8 = i & 15;
    const uint4 v = *reinterpret_cast<const uint4*>(q + ((size_t)b * HQ + hq) * HYQ_D + 8 * c8);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(lay.q_ring) +
                              (((size_t)b * HQ + hq) * period + pos) * HYQ_D + 8 * c8) = v;
  }
  for (int i = tid; i < HKV * HYQ_D / 8; i += blockDim.x) {
    const int hk = i >> 4, c8 = i & 15;
    const size_t bhk = (size_t)b * HKV + hk;
    const uint4 kv = *reinterpret_cast<const uint4*>(k_new + bhk * HYQ_D + 8 * c8);
    const uint4 vv = *reinterpret_cast<const uint4*>(v_new + bhk * HYQ_D + 8 * c8);
    const size_t to = (bhk * cap_tail + ntail) * HYQ_D + 8 * c8;
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(lay.tail_k) + to) = kv;
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(lay.tail_v) + to) = vv;
    if (k_src) {
      const size_t so = (bhk * ld + len) * HYQ_D + 8 * c8;
      *reinterpret_cast<uint4*>(k_src + so) = kv;
      *reinterpret_cast<uint4*>(v_src + so) = vv;
    }
  }
  __syncthreads();
  if (tid == 0) {
    cnt[HYQ_CNT_NTAIL] = ntail + 1;
    cnt[HYQ_CNT_LEN] = len + 1;
    cnt[HYQ_CNT_RING_POS] = (pos + 1) % period;
    cnt[HYQ_CNT_RING_N] = min(cnt[HYQ_CNT_RING_N] + 1, period);
  }
}

}  // namespace

size_t hyq_decode_ws_bytes(const hyq_config* c, int32_t len_hint) {
  // Enough for the global merge at the plan's split count (the fallback when
  // a cluster cannot be resident); the cluster and direct merges use none.
  const DecodePlan p = decode_plan(c, len_hint, false);  // the larger of the two plans
  size_t bh = (size_t)c->batch * c->num_kv_heads;
  return round_up(bh * 4) + round_up((size_t)c->batch * 4) + round_up(bh * (size_t)p.S * HYQ_MAX_GQA * kPart * 4);
}

template <int kMode, int BK, int BV>
cudaError_t set_attrs() {
  static std::atomic<uint64_t> done{0};
  return hyq_once_per_device(done, [] {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<kMode, BK, BV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Dec<BK, BV>::kSmemBytes);
    if (e == cudaSuccess && kMode == kCluster)
      e = cudaFuncSetAttribute(decode_kernel<kMode, BK, BV>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
  });
}

// Can one cluster of S decode blocks be resident on the current device?
// Cached per device (0 unknown, 1 yes, 2 no).
bool cluster_fits(int S) {
  static std::atomic<uint8_t> cached[kMaxDevices][17];
  if (S < 2 || S > 16) return false;
  const int dev = hyq_device();
  if (dev >= 0) {
    const uint8_t c = cached[dev][S].load(std::memory_order_relaxed);
    if (c) return c == 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Dec<4, 4>::kSmemBytes;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = S;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  bool ok = cudaOccupancyMaxActiveClusters(&n, decode_kernel<kCluster, 4, 4>, &cfg) == cudaSuccess && n >= 1;
  cudaGetLastError();
  if (dev >= 0) cached[dev][S].store(ok ? 1 : 2, std::memory_order_relaxed);
  return ok;
}

extern "C" hyq_status hyq_set_decode_overlap(int32_t enable) {
  if (enable != 0 && enable != 1) return HYQ_ERR_INVALID_ARG;
  g_overlap.store(enable, std::memory_order_relaxed);
  return HYQ_OK;
}

extern "C" hyq_status hyq_set_decode_plan(int32_t merge, int32_t splits) {
  if (merge < 0 || merge > 3) return HYQ_ERR_INVALID_ARG;
  if (merge == 2 && (splits < 2 || splits > 16)) return HYQ_ERR_INVALID_ARG;
  if (merge == 3 && (splits < 1 || splits > kMaxSplits)) return HYQ_ERR_INVALID_ARG;
  g_plan.store((merge << 16) | (merge == 0 ? 0 : splits), std::memory_order_relaxed);
  return HYQ_OK;
}

cudaError_t hyq_launch_decode(const hyq_config* c, const void* q, const hyq_layout* lay, void* out,
                              int32_t len_hint, void* ws, cudaStream_t s, const void* k_new, const void* v_new,
                              void* k_src, void* v_src, int32_t ld, const hyq_layout* next) {
  const int bk = hyq_bits_k(c), bv = hyq_bits_v(c);
  const bool w44 = bk == 4 && bv == 4;
  if (w44) {
    cudaError_t e = set_attrs<kCluster, 4, 4>();
    if (e != cudaSuccess) return e;
  }
  const int32_t overlap = g_overlap.load(std::memory_order_relaxed);
  DecodePlan p = decode_plan(c, len_hint, overlap != 0);
  // Cluster merge: 4-bit codes only, and only when the clusters fit; else the
  // workspace merge with the same S.
  if (p.mode == kCluster && (!w44 || !cluster_fits(p.S))) p.mode = kGlobal;
  size_t bh = (size_t)c->batch * c->num_kv_heads;
  int32_t* tickets = static_cast<int32_t*>(ws);
  StepArgs sa{static_cast<const __nv_bfloat16*>(k_new),
              static_cast<const __nv_bfloat16*>(v_new),
              static_cast<__nv_bfloat16*>(k_src),
              static_cast<__nv_bfloat16*>(v_src),
              ld,
              c->period,
              reinterpret_cast<int32_t*>(static_cast<char*>(ws) + round_up(bh * 4)),
              overlap,
              next ? next->qblocks : nullptr,
              next ? next->counts : nullptr,
              next ? static_cast<const __nv_bfloat16*>(next->vl_k) : nullptr,
              next ? static_cast<const __nv_bfloat16*>(next->vl_v) : nullptr,
              next ? static_cast<const __nv_bfloat16*>(next->tail_k) : nullptr,
              next ? static_cast<const __nv_bfloat16*>(next->tail_v) : nullptr};
  float* part = reinterpret_cast<float*>(static_cast<char*>(ws) + round_up(bh * 4) + round_up((size_t)c->batch * 4));
  const int gq = c->num_q_heads / c->num_kv_heads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.S, c->num_kv_heads, c->batch);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = p.S;
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;
  cfg.attrs = overlap ? attrs : attrs + 1;
  cfg.numAttrs = overlap ? 1 : 0;
  const __nv_bfloat16* qq = static_cast<const __nv_bfloat16*>(q);
  __nv_bfloat16* oo = static_cast<__nv_bfloat16*>(out);
  const int nblk = hyq_nblk(c), cvl = hyq_vl_stride(c), ct = hyq_cap_tail(c);
  // Launch one instantiation with its shared-memory plan.
  auto go = [&](auto kern, int smem_bytes, cudaError_t attr_err) {
    if (attr_err != cudaSuccess) return attr_err;
    cfg.dynamicSmemBytes = smem_bytes;
    return cudaLaunchKernelEx(&cfg, kern, qq, *lay, oo, tickets, part, c->num_q_heads, gq, nblk, cvl, ct, p.S, sa);
  };
  if (p.mode == kCluster) {  // 4-bit codes only (above)
    cfg.numAttrs += 1;
    return go(decode_kernel<kCluster, 4, 4>, Dec<4, 4>::kSmemBytes, cudaSuccess);
  }
  const bool direct = p.mode == kDirect;
  if (w44)
    return direct ? go(decode_kernel<kDirect, 4, 4>, Dec<4, 4>::kSmemBytes, set_attrs<kDirect, 4, 4>())
                  : go(decode_kernel<kGlobal, 4, 4>, Dec<4, 4>::kSmemBytes, set_attrs<kGlobal, 4, 4>());
  if (bk == 8 && bv == 8)
    return direct ? go(decode_kernel<kDirect, 8, 8>, Dec<8, 8>::kSmemBytes, set_attrs<kDirect, 8, 8>())
                  : go(decode_kernel<kGlobal, 8, 8>, Dec<8, 8>::kSmemBytes, set_attrs<kGlobal, 8, 8>());
  if (bk == 4)
    return direct ? go(decode_kernel<kDirect, 4, 8>, Dec<4, 8>::kSmemBytes, set_attrs<kDirect, 4, 8>())
                  : go(decode_kernel<kGlobal, 4, 8>, Dec<4, 8>::kSmemBytes, set_attrs<kGlobal, 4, 8>());
  return direct ? go(decode_kernel<kDirect, 8, 4>, Dec<8, 4>::kSmemBytes, set_attrs<kDirect, 8, 4>())
                : go(decode_kernel<kGlobal, 8, 4>, Dec<8, 4>::kSmemBytes, set_attrs<kGlobal, 8, 4>());
}

cudaError_t hyq_launch_decode_append(const hyq_config* c, const void* q, const void* k_new,
                                     const void* v_new, const hyq_layout* lay, void* k_src,
                                     void* v_src, int32_t ld, cudaStream_t s) {
  decode_append_kernel<<<c->batch, 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k_new),
      static_cast<const __nv_bfloat16*>(v_new), *lay, static_cast<__nv_bfloat16*>(k_src),
      static_cast<__nv_bfloat16*>(v_src), ld, c->num_q_heads, c->num_kv_heads, c->period, hyq_cap_tail(c));
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Decode attention for callers that cannot allocate device memory: the split
// partials and tickets live in this library-owned array instead of a
// caller-provided workspace.  Host code never dereferences the symbol; it
// looks up the array's device address once per device and passes that.
// ---------------------------------------------------------------------------
#include <mutex>

static __device__ __align__(256) unsigned char g_hyq_noalloc_scratch[HYQ_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[kMaxDevices] = {};

bool ptr_ok(const void* p, size_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) == 0; }
}  // namespace

extern "C" hyq_status hyq_decode_attention_noalloc(const hyq_config* c, const void* q,
                                                   const hyq_layout* l, void* out, int32_t len_hint,
                                                   hyq_stream_t s) {
  hyq_status st = hyq_config_check(c);
  if (st != HYQ_OK) return st;
  if (!l || !ptr_ok(q, 16) || !ptr_ok(out, 16) || len_hint < 0) return HYQ_ERR_INVALID_ARG;
  const void* ps[] = {l->qblocks, l->vl_k, l->vl_v, l->vl_idx, l->tail_k, l->tail_v, l->q_ring,
                      l->counts, l->err};
  for (const void* p : ps)
    if (!ptr_ok(p, 256)) return HYQ_ERR_INVALID_ARG;
  if (len_hint == 0 || len_hint > c->capacity) len_hint = c->capacity;
  if (hyq_decode_ws_bytes(c, len_hint) > HYQ_NOALLOC_SCRATCH_BYTES) return HYQ_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return HYQ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return HYQ_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_hyq_noalloc_scratch) != cudaSuccess || !p) return HYQ_ERR_CUDA;
      g_noalloc_addr[dev] = p;
    }
    scratch = g_noalloc_addr[dev];
  }
  // The tickets at the front of the scratch must start at zero.
  const size_t tickets = (size_t)c->batch * c->num_kv_heads * sizeof(int32_t);
  if (cudaMemsetAsync(scratch, 0, tickets, s) != cudaSuccess) return HYQ_ERR_CUDA;
  return hyq_launch_decode(c, q, l, out, len_hint, scratch, s) == cudaSuccess ? HYQ_OK : HYQ_ERR_CUDA;
}
