// Internal helpers shared by the libhyq kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/hyq.h"

#define HYQ_D 128
#define HYQ_G 32
#define HYQ_NGROUPS 4
#define HYQ_MAX_GQA 8
#define HYQ_TILE_BYTES 1024
#define HYQ_KMETA_OFF 8192
#define HYQ_VMETA_OFF 9216
#define HYQ_VCODE_OFF 4096

// ---------------------------------------------------------------------------
// Launch plumbing shared by the translation units (defined in hyq_api.cu).
// ---------------------------------------------------------------------------
// Devices the per-device host caches cover (device ordinals 0 .. kMaxDevices-1).
constexpr int kMaxDevices = 64;
int hyq_num_sms();
// Ordinal of the current device, or -1 when it cannot be read or lies past kMaxDevices.
inline int hyq_device() {
  int d = 0;
  return cudaGetDevice(&d) == cudaSuccess && d >= 0 && d < kMaxDevices ? d : -1;
}
// Runs f() (an idempotent setup returning cudaError_t, e.g. a kernel attribute)
// until it has succeeded once with the current device; `done` holds one bit
// per device.  Two threads making the first call at once may both run f.
template <class F>
cudaError_t hyq_once_per_device(std::atomic<uint64_t>& done, F f) {
  const int d = hyq_device();
  if (d < 0) return f();
  const uint64_t bit = 1ull << d;
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  const cudaError_t e = f();
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}
int32_t hyq_cap_vl(const hyq_config* c);
inline int32_t hyq_cap_tail(const hyq_config* c) { return c->window + c->period; }
// Row stride of the vertical-line buffers (at least one row is allocated).
inline int32_t hyq_vl_stride(const hyq_config* c) { return hyq_cap_vl(c) > 0 ? hyq_cap_vl(c) : 1; }
inline int32_t hyq_nblk(const hyq_config* c) { return (c->capacity + HYQ_QBLOCK_ROWS - 1) / HYQ_QBLOCK_ROWS; }
// Code widths B_K / B_V (a zero field means 4) and the stream's block size.
inline int hyq_bits_k(const hyq_config* c) { return c->bits_k == 0 ? 4 : c->bits_k; }
inline int hyq_bits_v(const hyq_config* c) { return c->bits_v == 0 ? 4 : c->bits_v; }
inline size_t hyq_qblock_bytes(const hyq_config* c) {
  return HYQ_QBLOCK_BYTES_BITS((size_t)hyq_bits_k(c), (size_t)hyq_bits_v(c));
}

// Byte layout of one 16-row quantised tile with B_K-bit keys and B_V-bit values.
template <int BK, int BV>
struct QFmt {
  static_assert((BK == 4 || BK == 8) && (BV == 4 || BV == 8), "code widths are 4 or 8 bits");
  static constexpr int kVCode = 256 * BK;        // K codes at 0, V codes here
  static constexpr int kKMeta = 256 * (BK + BV);  // K (scale, zero) pairs
  static constexpr int kVMeta = kKMeta + 256;     // V (scale, zero) pairs
  static constexpr int kTile = HYQ_QTILE_BYTES_BITS(BK, BV);
  static constexpr int kBlock = 4 * kTile;
};

// Kernel launchers (return the launch's cudaError_t).
cudaError_t hyq_launch_age_tail(const hyq_config* c, const hyq_layout* lay, cudaStream_t s);
cudaError_t hyq_launch_quantize_append(const hyq_config* c, const void* k, const void* v,
                                       int32_t n_rows, const hyq_layout* lay, cudaStream_t s);
cudaError_t hyq_launch_rebuild(const hyq_config* c, const void* k_src, const void* v_src,
                               int32_t ld, int32_t L, const int32_t* idx, int32_t k,
                               const hyq_layout* lay, cudaStream_t s);
cudaError_t hyq_launch_select(const hyq_config* c, const void* q_proxy, int32_t n_proxy,
                              int32_t n_proxy_ld, const void* k_src, int32_t ld, int32_t L,
                              int32_t* idx_out, int32_t k, void* ws, cudaStream_t s);
size_t hyq_select_ws_bytes(const hyq_config* c, int32_t L);
size_t hyq_select_kv_ws_bytes(const hyq_config* c, int32_t L);
// Vertical-line count of one query head (Algorithm 1's k) for a prefix of P.
int32_t hyq_vl_count_head(const hyq_config* c, int32_t P);
cudaError_t hyq_launch_select_heads(const hyq_config* c, const void* q_proxy, int32_t n_proxy,
                                    int32_t n_proxy_ld, const void* k_src, int32_t ld, int32_t L,
                                    int32_t* idx_heads, int32_t k1, int32_t* idx_out, int32_t ku, void* ws,
                                    cudaStream_t s);
size_t hyq_select_mass_ws_bytes(const hyq_config* c, int32_t L);
cudaError_t hyq_launch_select_mass(const hyq_config* c, const void* q_proxy, int32_t n_proxy,
                                   int32_t n_proxy_ld, const void* k_src, int32_t ld, int32_t L,
                                   int32_t* idx_out, int32_t k, void* ws, cudaStream_t s);
cudaError_t hyq_launch_decode_append(const hyq_config* c, const void* q, const void* k_new,
                                     const void* v_new, const hyq_layout* lay, void* k_src,
                                     void* v_src, int32_t ld, cudaStream_t s);
// k_new != nullptr: the fused step (append this token, then attend).
cudaError_t hyq_launch_decode(const hyq_config* c, const void* q, const hyq_layout* lay,
                              void* out, int32_t len_hint, void* ws, cudaStream_t s,
                              const void* k_new = nullptr, const void* v_new = nullptr,
                              void* k_src = nullptr, void* v_src = nullptr, int32_t ld = 0,
                              const hyq_layout* next = nullptr);
size_t hyq_decode_ws_bytes(const hyq_config* c, int32_t len_hint);
cudaError_t hyq_launch_prefill(const hyq_config* c, int dtype, const void* q, int64_t ldq, const void* k,
                               const void* v, int64_t ldk, int32_t L, const int32_t* vl, int32_t kvl, void* out,
                               void* ws, int32_t* err, cudaStream_t s, bool band);
size_t hyq_prefill_ws_bytes(const hyq_config* c, int dtype, int32_t L, int32_t kvl, bool band);
size_t hyq_prefill_ws_bytes_hint(const hyq_config* c, int32_t L, bool band);

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void hyq_set_err(int32_t* err, int32_t bits) {
  if (err) atomicOr(err, bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D += A * B, m16n8k16, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose an 8x8 b16 matrix held one row-pair per thread.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(a));
  return d;
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                                  uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Two 4-bit codes (nibbles sh and sh+16 of w) as a bf16 pair (128 + c).
__device__ __forceinline__ uint32_t nib2_bf16(uint32_t w, int sh) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;\n" : "=r"(r) : "r"(w >> sh), "r"(0x000F000Fu), "r"(0x43004300u));
  return r;
}

// Two 4-bit codes as an fp16 pair of subnormals c * 2^-24 (exact; the tensor
// cores take fp16 subnormal operands at full precision).  Unlike an offset
// encoding there is nothing to cancel afterwards, so rounding the other
// operand to fp16 does not get amplified.
__device__ __forceinline__ uint32_t nib2_f16_sub(uint32_t w, int sh) {
  return (w >> sh) & 0x000F000Fu;
}
#define HYQ_F16_SUB_SCALE 16777216.0f  // 2^24: undoes the subnormal code scale

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float2 half2_to_float2(uint32_t u) {
  __half2 h = *reinterpret_cast<__half2*>(&u);
  return __half22float2(h);
}

// ----- mbarrier + bulk copy (non-tensor TMA) -------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::);
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Bounded wait for the given phase parity; returns false if it gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  uint32_t addr = smem_u32(bar);
  for (int it = 0; it < (1 << 22); ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// Global -> shared bulk copy (16-byte aligned addresses, size a multiple of 16),
// completion counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ float warp_max_xor(float v, int lanemask_start) {
  for (int o = lanemask_start; o < 32; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
