// Hybrid-precision decode attention ("HyQuant: Hybrid-Precision Quantization
// for LLM Attention", §4.3 Eq. 8-9 and Appendix A.3 Algorithm 3) and the
// per-step bookkeeping (append to the BF16 tail, proxy-query ring of §5.5).
//
// Work decomposition (one launch):
//   grid.x = S_q + S_f thread blocks per (batch, KV head).  The first S_q
//   blocks split the 4-bit stream along the sequence (Algorithm 3, segment 1
//   "partition K^Q into S chunks"); the last S_f split the BF16 rows
//   (vertical-line rows, then the tail).  Every block keeps one online
//   softmax state (m, l, acc) per query head of the KV group (the g query
//   heads are packed into one tensor-core tile, Algorithm 3 line "pack g GQA
//   heads"), writes it to the workspace, and the last block to finish (an
//   atomic ticket; nobody waits) merges all partials by log-sum-exp
//   rescaling (ReduceSoftmax) and writes the BF16 output.
//
// 4-bit tiles (16 rows) are dequantised inside the dot products:
//   q.k~  = sum_q s_q (q_q . c_q) + z_q sum(q_q)     (per group q of 32)
//   p v~  = sum_j (p_j s_jq) c_jd + p_j z_jq
// The code products run on mma.sync m16n8k16 with the codes unpacked from
// nibbles into register pairs by one lop3/and each: K codes as bf16 128 + c
// (the offset is removed exactly through the per-group query sums, since q
// and s enter unrounded), V codes as fp16 subnormals c * 2^-24 against the
// fp16-rounded p * s (no offset, so the rounding of p * s is not amplified).
// Scale/zero terms are applied in fp32.
#include <math.h>

#include "hyq_common.cuh"

namespace {

constexpr int kThreads = 128;  // 4 warps, one 16-row tile each
constexpr int kWarps = 4;
constexpr int kQStages = 4;      // 4-bit blocks in flight per CTA
constexpr int kFRows = 64;       // BF16 rows per stage
constexpr int kFStride = 272;    // padded BF16 row in shared memory (conflict-free ldmatrix)
constexpr int kFStages = 2;
constexpr int kStageFBytes = 2 * kFRows * kFStride;
constexpr int kSmemBytes = (kQStages * HYQ_QBLOCK_BYTES > kFStages * kStageFBytes)
                               ? kQStages * HYQ_QBLOCK_BYTES
                               : kFStages * kStageFBytes;
constexpr int kPart = 2 + HYQ_D;  // m, l, acc[128] per head
constexpr int kMaxSplits = 512;
// log2(e) / sqrt(128): logits are kept in the base-2 domain.
constexpr float kScale = 0.1275174307366466f;

size_t round_up(size_t x) { return (x + 255) / 256 * 256; }

void decode_split(const hyq_config* c, int32_t len, int& sq, int& sf) {
  const int bh = c->batch * c->num_kv_heads;
  const int target = 2 * hyq_num_sms();
  int per_bh = (target + bh - 1) / bh;
  if (per_bh < 2) per_bh = 2;
  int32_t P = len - c->window > 0 ? len - c->window : 0;
  int32_t nvl = hyq_vl_count(c, P);
  int64_t nq = P - nvl;
  int64_t nf = (int64_t)nvl + (len < hyq_cap_tail(c) ? len : hyq_cap_tail(c));
  double bq = 160.0 * nq, bf = 512.0 * nf;
  sq = (int)(per_bh * bq / (bq + bf + 1.0) + 0.5);
  int sq_max = (int)((nq + HYQ_QBLOCK_ROWS - 1) / HYQ_QBLOCK_ROWS);
  if (sq > sq_max) sq = sq_max;
  if (sq < 1) sq = 1;
  sf = per_bh - sq;
  int sf_max = (int)((nf + 2 * 16 - 1) / (2 * 16));  // at least ~32 rows per block
  if (sf > sf_max) sf = sf_max;
  if (sf < 1) sf = 1;
  if (sq + sf > kMaxSplits) {
    sq = kMaxSplits - sf;
  }
}

struct State {
  float m[2], l[2];
  float acc[8][4];
  float zacc[2][4];
};

// Online-softmax update of the two heads (2t, 2t+1) this thread owns with the
// logits of tokens (g, g+8); returns the probabilities p[2r + j].
__device__ __forceinline__ void softmax_update(const float (&lg)[4], State& st, float (&p)[4]) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float tm = fmaxf(lg[j], lg[2 + j]);
    tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 4));
    tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 8));
    tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 16));
    const float mn = fmaxf(st.m[j], tm);
    const float ms = (mn == -INFINITY) ? 0.f : mn;
    const float corr = exp2f(st.m[j] - ms);
    p[j] = exp2f(lg[j] - ms);
    p[2 + j] = exp2f(lg[2 + j] - ms);
    st.l[j] = fmaf(st.l[j], corr, p[j] + p[2 + j]);
    st.m[j] = mn;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      st.acc[mt][j] *= corr;
      st.acc[mt][2 + j] *= corr;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) st.zacc[j][q] *= corr;
  }
}

// One 16-row tile of a 4-bit block (stage base `sb`, tile `w`), `vr` valid rows.
__device__ __forceinline__ void q_tile(const uint8_t* sb, int w, int lane, int vr,
                                       const uint32_t (&bq)[8][2], const float (&qs)[2][4],
                                       State& st) {
  const int g = lane >> 2;
  const uint8_t* kt = sb + w * HYQ_TILE_BYTES;
  const uint4 kw0 = *reinterpret_cast<const uint4*>(kt + lane * 16);
  const uint4 kw1 = *reinterpret_cast<const uint4*>(kt + 512 + lane * 16);
  const uint32_t kw[8] = {kw0.x, kw0.y, kw0.z, kw0.w, kw1.x, kw1.y, kw1.z, kw1.w};
  float C[4][4];
#pragma unroll
  for (int q = 0; q < 4; ++q) C[q][0] = C[q][1] = C[q][2] = C[q][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
    mma_bf16(C[ks >> 1], nib2_bf16(kw[ks], 0), nib2_bf16(kw[ks], 4), nib2_bf16(kw[ks], 8),
             nib2_bf16(kw[ks], 12), bq[ks][0], bq[ks][1]);
  const uint8_t* km = sb + HYQ_KMETA_OFF + w * 16 * 16;
  float lg[4];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const uint4 mk = *reinterpret_cast<const uint4*>(km + (g + 8 * r) * 16);
    const uint32_t mw[4] = {mk.x, mk.y, mk.z, mk.w};
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 sz = half2_to_float2(mw[q]);
      const float zz = fmaf(-128.f, sz.x, sz.y);  // zero minus the bf16 code offset
      a0 = fmaf(sz.x, C[q][2 * r], a0);
      a0 = fmaf(zz, qs[0][q], a0);
      a1 = fmaf(sz.x, C[q][2 * r + 1], a1);
      a1 = fmaf(zz, qs[1][q], a1);
    }
    const bool valid = g + 8 * r < vr;
    lg[2 * r] = valid ? a0 * kScale : -INFINITY;
    lg[2 * r + 1] = valid ? a1 * kScale : -INFINITY;
  }
  float p[4];
  softmax_update(lg, st, p);
  const uint8_t* vt = sb + HYQ_VCODE_OFF + w * HYQ_TILE_BYTES;
  const uint4 vw0 = *reinterpret_cast<const uint4*>(vt + lane * 16);
  const uint4 vw1 = *reinterpret_cast<const uint4*>(vt + 512 + lane * 16);
  const uint32_t vw[8] = {vw0.x, vw0.y, vw0.z, vw0.w, vw1.x, vw1.y, vw1.z, vw1.w};
  const uint8_t* vm = sb + HYQ_VMETA_OFF + w * 16 * 16;
  const uint4 mv0 = *reinterpret_cast<const uint4*>(vm + g * 16);
  const uint4 mv1 = *reinterpret_cast<const uint4*>(vm + (g + 8) * 16);
  const uint32_t m0[4] = {mv0.x, mv0.y, mv0.z, mv0.w};
  const uint32_t m1[4] = {mv1.x, mv1.y, mv1.z, mv1.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 sz0 = half2_to_float2(m0[q]);
    const float2 sz1 = half2_to_float2(m1[q]);
    // B operand (tokens x heads) of group q: p * s, transposed into place.
    const uint32_t b0 = movmatrix_trans(pack_f16x2(p[0] * sz0.x, p[1] * sz0.x));
    const uint32_t b1 = movmatrix_trans(pack_f16x2(p[2] * sz1.x, p[3] * sz1.x));
    st.zacc[0][q] = fmaf(p[0], sz0.y, fmaf(p[2], sz1.y, st.zacc[0][q]));
    st.zacc[1][q] = fmaf(p[1], sz0.y, fmaf(p[3], sz1.y, st.zacc[1][q]));
#pragma unroll
    for (int mm = 0; mm < 2; ++mm) {
      const uint32_t x = vw[2 * q + mm];
      // codes as c * 2^-24: acc collects 2^-24 * sum_j (p_j s_j) c_jd
      mma_f16(st.acc[2 * q + mm], nib2_f16_sub(x, 0), nib2_f16_sub(x, 4), nib2_f16_sub(x, 8),
              nib2_f16_sub(x, 12), b0, b1);
    }
  }
}

// One 16-row tile of BF16 rows (K rows at Ks, V rows at Vs, padded stride).
__device__ __forceinline__ void f_tile(const uint8_t* Ks, const uint8_t* Vs, int w, int lane, int vr,
                                       const uint32_t (&bq)[8][2], State& st) {
  const int g = lane >> 2, i4 = lane >> 3, rr = lane & 7;
  float S[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    uint32_t a0, a1, a2, a3;
    ldmatrix_x4(smem_u32(Ks + (w * 16 + rr + 8 * (i4 & 1)) * kFStride + (16 * ks + 8 * (i4 >> 1)) * 2), a0,
                a1, a2, a3);
    mma_bf16(S, a0, a1, a2, a3, bq[ks][0], bq[ks][1]);
  }
  float lg[4];
  lg[0] = g < vr ? S[0] * kScale : -INFINITY;
  lg[1] = g < vr ? S[1] * kScale : -INFINITY;
  lg[2] = g + 8 < vr ? S[2] * kScale : -INFINITY;
  lg[3] = g + 8 < vr ? S[3] * kScale : -INFINITY;
  float p[4];
  softmax_update(lg, st, p);
  const uint32_t b0 = movmatrix_trans(pack_bf16x2(p[0], p[1]));
  const uint32_t b1 = movmatrix_trans(pack_bf16x2(p[2], p[3]));
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    uint32_t a0, a1, a2, a3;
    ldmatrix_x4_trans(smem_u32(Vs + (w * 16 + rr + 8 * (i4 >> 1)) * kFStride + (16 * mt + 8 * (i4 & 1)) * 2),
                      a0, a1, a2, a3);
    mma_bf16(st.acc[mt], a0, a1, a2, a3, b0, b1);
  }
}

__global__ void __launch_bounds__(kThreads) decode_kernel(
    const __nv_bfloat16* __restrict__ q, hyq_layout lay, __nv_bfloat16* __restrict__ out,
    int32_t* __restrict__ tickets, float* __restrict__ part, int HQ, int gq, int nblk_cap,
    int cap_vl, int cap_tail, int S_q, int S_f) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(16) __nv_bfloat16 q_s[HYQ_MAX_GQA * HYQ_D];
  __shared__ float qsum_s[HYQ_MAX_GQA * 4];
  __shared__ __align__(8) uint64_t bars[kQStages];
  __shared__ int s_flag;

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z, HKV = gridDim.y;
  const int S_tot = S_q + S_f;
  const size_t bh = (size_t)b * HKV + h;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;

  const int32_t* cnt = lay.counts + (size_t)b * HYQ_COUNTS;
  int32_t nq = cnt[HYQ_CNT_NQ], nvl = cnt[HYQ_CNT_NVL], ntail = cnt[HYQ_CNT_NTAIL];
  if (nq < 0 || nq > nblk_cap * HYQ_QBLOCK_ROWS || nvl < 0 || nvl > cap_vl || ntail < 0 || ntail > cap_tail) {
    if (tid == 0 && split == 0) hyq_set_err(lay.err, HYQ_DEVERR_COUNT);
    nq = min(max(nq, 0), nblk_cap * HYQ_QBLOCK_ROWS);
    nvl = min(max(nvl, 0), cap_vl);
    ntail = min(max(ntail, 0), cap_tail);
  }

  // Query tile of the KV group (rows past g are zero) and its per-group sums.
  for (int i = tid; i < HYQ_MAX_GQA * HYQ_D / 8; i += kThreads) {
    const int row = i >> 4, c8 = i & 15;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < gq) v = *reinterpret_cast<const uint4*>(q + ((size_t)b * HQ + (size_t)h * gq + row) * HYQ_D + 8 * c8);
    *reinterpret_cast<uint4*>(q_s + row * HYQ_D + 8 * c8) = v;
  }
  if (tid == 0) {
    for (int i = 0; i < kQStages; ++i) mbar_init(&bars[i], 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (tid < 32) {
    float s = 0.f;
    const __nv_bfloat16* r = q_s + (tid >> 2) * HYQ_D + 32 * (tid & 3);
    for (int i = 0; i < 32; ++i) s += __bfloat162float(r[i]);
    qsum_s[tid] = s;
  }
  __syncthreads();
  uint32_t bq[8][2];
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    bq[ks][0] = *reinterpret_cast<const uint32_t*>(q_s + g * HYQ_D + 16 * ks + 2 * t);
    bq[ks][1] = *reinterpret_cast<const uint32_t*>(q_s + g * HYQ_D + 16 * ks + 2 * t + 8);
  }
  float qs[2][4];
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) qs[j][qq] = qsum_s[(2 * t + j) * 4 + qq];

  State st;
  st.m[0] = st.m[1] = -INFINITY;
  st.l[0] = st.l[1] = 0.f;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) st.acc[mt][0] = st.acc[mt][1] = st.acc[mt][2] = st.acc[mt][3] = 0.f;
#pragma unroll
  for (int j = 0; j < 2; ++j) st.zacc[j][0] = st.zacc[j][1] = st.zacc[j][2] = st.zacc[j][3] = 0.f;

  bool timed_out = false;
  int pend_lo = 0, pend_hi = 0, pend_stages = 1;  // copies still in flight after a timeout
  if (split < S_q) {
    // ---- 4-bit stream: blocks [b0, b1) of this split ----------------------
    const int nb = (nq + HYQ_QBLOCK_ROWS - 1) / HYQ_QBLOCK_ROWS;
    const int b0 = (int)((int64_t)split * nb / S_q), b1 = (int)((int64_t)(split + 1) * nb / S_q);
    const int n = b1 - b0;
    const uint8_t* src = lay.qblocks + (bh * nblk_cap + b0) * (size_t)HYQ_QBLOCK_BYTES;
    if (tid == 0) {
      for (int i = 0; i < n && i < kQStages; ++i) {
        mbar_arrive_expect_tx(&bars[i], HYQ_QBLOCK_BYTES);
        bulk_g2s(smem + i * HYQ_QBLOCK_BYTES, src + (size_t)i * HYQ_QBLOCK_BYTES, HYQ_QBLOCK_BYTES, &bars[i]);
      }
    }
    for (int i = 0; i < n; ++i) {
      const int sidx = i % kQStages;
      const bool ok = mbar_wait(&bars[sidx], (i / kQStages) & 1);
      if (__syncthreads_or(!ok)) {
        timed_out = true;
        pend_lo = i;
        pend_hi = min(n, i + kQStages);
        pend_stages = kQStages;
        break;
      }
      const int vr = min(HYQ_QBLOCK_ROWS, nq - (b0 + i) * HYQ_QBLOCK_ROWS) - 16 * warp;
      if (vr > 0) q_tile(smem + sidx * HYQ_QBLOCK_BYTES, warp, lane, vr, bq, qs, st);
      __syncthreads();
      if (tid == 0 && i + kQStages < n) {
        mbar_arrive_expect_tx(&bars[sidx], HYQ_QBLOCK_BYTES);
        bulk_g2s(smem + sidx * HYQ_QBLOCK_BYTES, src + (size_t)(i + kQStages) * HYQ_QBLOCK_BYTES,
                 HYQ_QBLOCK_BYTES, &bars[sidx]);
      }
    }
  } else {
    // ---- BF16 rows: vertical-line rows then tail rows ----------------------
    const int nf = nvl + ntail;
    const int sp = split - S_q;
    const int r0 = (int)((int64_t)sp * nf / S_f), r1 = (int)((int64_t)(sp + 1) * nf / S_f);
    const int nst = (r1 - r0 + kFRows - 1) / kFRows;
    // Rows past the copied count must hold finite values: zero the stages once.
    for (int i = tid; i < kFStages * kStageFBytes / 16; i += kThreads)
      reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    __syncthreads();
    const __nv_bfloat16* vlk = static_cast<const __nv_bfloat16*>(lay.vl_k) + bh * cap_vl * HYQ_D;
    const __nv_bfloat16* vlv = static_cast<const __nv_bfloat16*>(lay.vl_v) + bh * cap_vl * HYQ_D;
    const __nv_bfloat16* tk = static_cast<const __nv_bfloat16*>(lay.tail_k) + bh * cap_tail * HYQ_D;
    const __nv_bfloat16* tv = static_cast<const __nv_bfloat16*>(lay.tail_v) + bh * cap_tail * HYQ_D;
    auto issue = [&](int stage, int rbase) {
      const int nrows = min(kFRows, r1 - rbase);
      uint8_t* Ks = smem + stage * kStageFBytes;
      uint8_t* Vs = Ks + kFRows * kFStride;
      if (lane == 0) mbar_arrive_expect_tx(&bars[stage], nrows * 2 * HYQ_D * 2);
      __syncwarp();
      for (int rr = lane; rr < nrows; rr += 32) {
        const int row = rbase + rr;
        const __nv_bfloat16* sk = row < nvl ? vlk + (size_t)row * HYQ_D : tk + (size_t)(row - nvl) * HYQ_D;
        const __nv_bfloat16* sv = row < nvl ? vlv + (size_t)row * HYQ_D : tv + (size_t)(row - nvl) * HYQ_D;
        bulk_g2s(Ks + rr * kFStride, sk, HYQ_D * 2, &bars[stage]);
        bulk_g2s(Vs + rr * kFStride, sv, HYQ_D * 2, &bars[stage]);
      }
    };
    if (warp == 0)
      for (int i = 0; i < nst && i < kFStages; ++i) issue(i, r0 + i * kFRows);
    for (int i = 0; i < nst; ++i) {
      const int sidx = i % kFStages;
      const bool ok = mbar_wait(&bars[sidx], (i / kFStages) & 1);
      if (__syncthreads_or(!ok)) {
        timed_out = true;
        pend_lo = i;
        pend_hi = min(nst, i + kFStages);
        pend_stages = kFStages;
        break;
      }
      const uint8_t* Ks = smem + sidx * kStageFBytes;
      const int vr = min(kFRows, r1 - (r0 + i * kFRows)) - 16 * warp;
      if (vr > 0) f_tile(Ks, Ks + kFRows * kFStride, warp, lane, vr, bq, st);
      __syncthreads();
      if (warp == 0 && i + kFStages < nst) issue(sidx, r0 + (i + kFStages) * kFRows);
    }
  }
  if (timed_out) {
    // A bulk copy did not arrive: report it and make sure none is still in
    // flight into this block's shared memory before the block exits.
    if (tid == 0) {
      hyq_set_err(lay.err, HYQ_DEVERR_TIMEOUT);
      for (int i = pend_lo; i < pend_hi; ++i) (void)mbar_wait(&bars[i % pend_stages], (i / pend_stages) & 1);
    }
    __syncthreads();
    return;
  }

  if (split < S_q) {  // the 4-bit PV products were taken on codes scaled by 2^-24
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int ci = 0; ci < 4; ++ci) st.acc[mt][ci] *= HYQ_F16_SUB_SCALE;
  }
  // ---- reduce the thread-partial sums over the 8 lanes sharing t ----------
#pragma unroll
  for (int j = 0; j < 2; ++j) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) st.l[j] += __shfl_xor_sync(0xffffffffu, st.l[j], o);
#pragma unroll
    for (int qq = 0; qq < 4; ++qq)
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) st.zacc[j][qq] += __shfl_xor_sync(0xffffffffu, st.zacc[j][qq], o);
  }
  __syncthreads();  // stage memory is free from here on
  float* red = reinterpret_cast<float*>(smem);           // [warp][head][128]
  float* red_m = red + kWarps * HYQ_MAX_GQA * HYQ_D;     // [warp][head]
  float* red_l = red_m + kWarps * HYQ_MAX_GQA;
  float* wts = red_l + kWarps * HYQ_MAX_GQA;             // [warp][head]
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int ci = 0; ci < 4; ++ci) {
      const int d = 16 * mt + g + 8 * (ci >> 1), hd = 2 * t + (ci & 1);
      red[(warp * HYQ_MAX_GQA + hd) * HYQ_D + d] = st.acc[mt][ci] + st.zacc[ci & 1][mt >> 1];
    }
  if (g == 0)
    for (int j = 0; j < 2; ++j) {
      red_m[warp * HYQ_MAX_GQA + 2 * t + j] = st.m[j];
      red_l[warp * HYQ_MAX_GQA + 2 * t + j] = st.l[j];
    }
  __syncthreads();
  float* pp = part + (bh * S_tot + split) * (size_t)(HYQ_MAX_GQA * kPart);
  if (tid < gq) {
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w * HYQ_MAX_GQA + tid]);
    const float Ms = (M == -INFINITY) ? 0.f : M;
    float Lsum = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      const float wt = exp2f(red_m[w * HYQ_MAX_GQA + tid] - Ms);
      wts[w * HYQ_MAX_GQA + tid] = wt;
      Lsum = fmaf(red_l[w * HYQ_MAX_GQA + tid], wt, Lsum);
    }
    pp[tid * kPart + 0] = M;
    pp[tid * kPart + 1] = Lsum;
  }
  __syncthreads();
  for (int i = tid; i < gq * HYQ_D; i += kThreads) {
    const int hd = i >> 7, d = i & (HYQ_D - 1);
    float a = 0.f;
    for (int w = 0; w < kWarps; ++w) a = fmaf(red[(w * HYQ_MAX_GQA + hd) * HYQ_D + d], wts[w * HYQ_MAX_GQA + hd], a);
    pp[hd * kPart + 2 + d] = a;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_flag = (atomicAdd(&tickets[bh], 1) == S_tot - 1);
  __syncthreads();
  if (!s_flag) return;
  __threadfence();

  // ---- last block: ReduceSoftmax over the S_tot partials -------------------
  const float* pb = part + bh * S_tot * (size_t)(HYQ_MAX_GQA * kPart);
  float* sM = red;                       // [head]
  float* sL = sM + HYQ_MAX_GQA;          // [head]
  float* sw = sL + HYQ_MAX_GQA;          // [split][head]
  if (tid < gq) {
    float M = -INFINITY;
    for (int s2 = 0; s2 < S_tot; ++s2) M = fmaxf(M, __ldcg(pb + (size_t)s2 * HYQ_MAX_GQA * kPart + tid * kPart));
    sM[tid] = (M == -INFINITY) ? 0.f : M;
  }
  __syncthreads();
  for (int i = tid; i < S_tot * gq; i += kThreads) {
    const int s2 = i / gq, hd = i % gq;
    const float* e = pb + (size_t)s2 * HYQ_MAX_GQA * kPart + hd * kPart;
    sw[s2 * HYQ_MAX_GQA + hd] = exp2f(__ldcg(e) - sM[hd]);
  }
  __syncthreads();
  if (tid < gq) {
    float Lsum = 0.f;
    for (int s2 = 0; s2 < S_tot; ++s2)
      Lsum = fmaf(__ldcg(pb + (size_t)s2 * HYQ_MAX_GQA * kPart + tid * kPart + 1), sw[s2 * HYQ_MAX_GQA + tid], Lsum);
    sL[tid] = Lsum;
  }
  __syncthreads();
  for (int i = tid; i < gq * HYQ_D; i += kThreads) {
    const int hd = i >> 7, d = i & (HYQ_D - 1);
    float a = 0.f;
    for (int s2 = 0; s2 < S_tot; ++s2)
      a = fmaf(__ldcg(pb + (size_t)s2 * HYQ_MAX_GQA * kPart + hd * kPart + 2 + d), sw[s2 * HYQ_MAX_GQA + hd], a);
    const float Lh = sL[hd];
    out[((size_t)b * HQ + (size_t)h * gq + hd) * HYQ_D + d] = __float2bfloat16_rn(Lh > 0.f ? a / Lh : 0.f);
  }
  if (tid == 0) tickets[bh] = 0;
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
  int sq, sf;
  decode_split(c, len_hint, sq, sf);
  size_t bh = (size_t)c->batch * c->num_kv_heads;
  return round_up(bh * 4) + round_up(bh * (size_t)(sq + sf) * HYQ_MAX_GQA * kPart * 4);
}

cudaError_t hyq_launch_decode(const hyq_config* c, const void* q, const hyq_layout* lay, void* out,
                              int32_t len_hint, void* ws, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  int sq, sf;
  decode_split(c, len_hint, sq, sf);
  size_t bh = (size_t)c->batch * c->num_kv_heads;
  int32_t* tickets = static_cast<int32_t*>(ws);
  float* part = reinterpret_cast<float*>(static_cast<char*>(ws) + round_up(bh * 4));
  dim3 grid(sq + sf, c->num_kv_heads, c->batch);
  decode_kernel<<<grid, kThreads, kSmemBytes, s>>>(
      static_cast<const __nv_bfloat16*>(q), *lay, static_cast<__nv_bfloat16*>(out), tickets, part,
      c->num_q_heads, c->num_q_heads / c->num_kv_heads, hyq_nblk(c), hyq_vl_stride(c), hyq_cap_tail(c), sq, sf);
  return cudaGetLastError();
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
constexpr int kMaxDevices = 64;
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
