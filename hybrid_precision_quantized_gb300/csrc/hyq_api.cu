// Host side of the libhyq C ABI: argument validation, buffer sizing and
// dispatch to the kernels.  Every check runs before any launch, so an invalid
// call leaves all buffers untouched.
#include <atomic>
#include <cstdint>
#include <cstring>

#include "hyq_common.cuh"

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

hyq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? HYQ_OK : HYQ_ERR_CUDA; }

// Every layout pointer is present and 256-byte aligned.
bool layout_ok(const hyq_layout* l) {
  if (!l) return false;
  const void* ps[] = {l->qblocks, l->vl_k, l->vl_v, l->vl_idx, l->tail_k, l->tail_v,
                      l->q_ring, l->counts, l->err};
  for (const void* p : ps)
    if (!p || !aligned(p, kAlign)) return false;
  return true;
}

}  // namespace

// Streaming-multiprocessor count of the current device, cached per device
// (atomics: any host thread may call this for any device).
int hyq_num_sms() {
  static std::atomic<int> cached[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) dev = -1;
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (dev < 0 || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev >= 0 && dev < kMaxDevices) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

extern "C" const char* hyq_status_string(hyq_status s) {
  switch (s) {
    case HYQ_OK: return "ok";
    case HYQ_ERR_INVALID_ARG: return "invalid argument";
    case HYQ_ERR_UNSUPPORTED: return "unsupported";
    case HYQ_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case HYQ_ERR_CAPACITY: return "length exceeds layout capacity";
    case HYQ_ERR_CUDA: return "CUDA error";
    case HYQ_ERR_DEVICE: return "device error word set";
  }
  return "unknown status";
}

extern "C" hyq_status hyq_config_check(const hyq_config* c) {
  if (!c) return HYQ_ERR_INVALID_ARG;
  if (c->batch < 1 || c->num_q_heads < 1 || c->num_kv_heads < 1) return HYQ_ERR_INVALID_ARG;
  if (c->num_q_heads % c->num_kv_heads) return HYQ_ERR_INVALID_ARG;
  int g = c->num_q_heads / c->num_kv_heads;
  if (g > HYQ_MAX_GQA) return HYQ_ERR_UNSUPPORTED;
  if (c->head_dim != HYQ_D || c->group != HYQ_G) return HYQ_ERR_UNSUPPORTED;
  if (c->window < 0 || c->period < 1 || c->period > 1024) return HYQ_ERR_INVALID_ARG;
  if (c->rho_ppm < 0 || c->rho_ppm > 1000000) return HYQ_ERR_INVALID_ARG;
  if (c->capacity < 1 || c->capacity > (1 << 30)) return HYQ_ERR_INVALID_ARG;
  if (c->batch > 65535 || c->num_kv_heads > 65535) return HYQ_ERR_INVALID_ARG;
  if ((c->bits_k != 0 && c->bits_k != 4 && c->bits_k != 8) || (c->bits_v != 0 && c->bits_v != 4 && c->bits_v != 8))
    return HYQ_ERR_UNSUPPORTED;
  if (c->vl_mode != HYQ_VL_PER_KV_HEAD && c->vl_mode != HYQ_VL_PER_QUERY_HEAD) return HYQ_ERR_INVALID_ARG;
  return HYQ_OK;
}

int32_t hyq_vl_count_head(const hyq_config* c, int32_t P) {
  if (P <= 0 || c->rho_ppm <= 0) return 0;
  int64_t k = ((int64_t)P * c->rho_ppm + 999999) / 1000000;  // exact ceil(P * rho)
  if (k < 1) k = 1;
  if (k > P) k = P;
  return (int32_t)k;
}

extern "C" int32_t hyq_vl_count(const hyq_config* c, int32_t P) {
  if (!c) return -1;
  const int64_t k = hyq_vl_count_head(c, P);
  if (c->vl_mode != HYQ_VL_PER_QUERY_HEAD || c->num_kv_heads < 1) return (int32_t)k;
  const int64_t ku = k * (c->num_q_heads / c->num_kv_heads);
  return (int32_t)(ku < P ? ku : P);
}

int32_t hyq_cap_vl(const hyq_config* c) {
  int32_t P = c->capacity - c->window;
  return hyq_vl_count(c, P > 0 ? P : 0);
}

extern "C" hyq_status hyq_layout_sizes(const hyq_config* c, size_t* out) {
  hyq_status st = hyq_config_check(c);
  if (st != HYQ_OK) return st;
  if (!out) return HYQ_ERR_INVALID_ARG;
  size_t bh = (size_t)c->batch * c->num_kv_heads;
  size_t cap_vl = hyq_vl_stride(c);
  size_t cap_tail = hyq_cap_tail(c);
  out[0] = round_up(bh * hyq_nblk(c) * hyq_qblock_bytes(c));
  out[1] = round_up(bh * cap_vl * HYQ_D * 2);
  out[2] = out[1];
  out[3] = round_up(bh * cap_vl * 4);
  out[4] = round_up(bh * cap_tail * HYQ_D * 2);
  out[5] = out[4];
  out[6] = round_up((size_t)c->batch * c->num_q_heads * c->period * HYQ_D * 2);
  out[7] = round_up((size_t)c->batch * HYQ_COUNTS * 4);
  out[8] = round_up(4);
  return HYQ_OK;
}

extern "C" size_t hyq_workspace_size(const hyq_config* c, int op, int32_t len_hint) {
  if (hyq_config_check(c) != HYQ_OK || len_hint < 0) return 0;
  if (len_hint == 0 || len_hint > c->capacity) len_hint = c->capacity;
  switch (op) {
    case HYQ_OP_SELECT: return hyq_select_ws_bytes(c, len_hint);
    case HYQ_OP_SELECT_MASS: return hyq_select_mass_ws_bytes(c, len_hint);
    case HYQ_OP_DECODE: return hyq_decode_ws_bytes(c, len_hint);
    case HYQ_OP_PREFILL: return hyq_prefill_ws_bytes_hint(c, len_hint, false);
    case HYQ_OP_PREFILL_BAND: return hyq_prefill_ws_bytes_hint(c, len_hint, true);
    default: return 0;
  }
}

extern "C" hyq_status hyq_layout_reset(const hyq_config* c, const hyq_layout* l, hyq_stream_t s) {
  hyq_status st = hyq_config_check(c);
  if (st != HYQ_OK) return st;
  if (!layout_ok(l)) return HYQ_ERR_INVALID_ARG;
  cudaError_t e = cudaMemsetAsync(l->counts, 0, (size_t)c->batch * HYQ_COUNTS * 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(l->err, 0, 4, s);
  return from_cuda(e);
}

extern "C" hyq_status hyq_quantize_append(const hyq_config* c, const void* k_rows,
                                          const void* v_rows, int32_t n_rows,
                                          const hyq_layout* l, hyq_stream_t s) {
  hyq_status st = hyq_config_check(c);
  if (st != HYQ_OK) return st;
  if (!layout_ok(l) || n_rows < 0) return HYQ_ERR_INVALID_ARG;
  if (n_rows == 0) return HYQ_OK;
  if (!k_rows || !v_rows || !aligned(k_rows, 16) || !aligned(v_rows, 16)) return HYQ_ERR_INVALID_ARG;
  if (n_rows > hyq_nblk(c) * HYQ_QBLOCK_ROWS) return HYQ_ERR_CAPACITY;
  return from_cuda(hyq_launch_quantize_append(c, k_rows, v_rows, n_rows, l, s));
}

extern "C" hyq_status hyq_age_tail(const hyq_config* c, const hyq_layout* l, hyq_stream_t s) {
  hyq_status st = hyq_config_check(c);
  if (st != HYQ_OK) return st;
  if (!layout_ok(l)) return HYQ_ERR_INVALID_ARG;
  return from_cuda(hyq_launch_age_tail(c, l, s));
}

extern "C" hyq_status hyq_select_vertical(const hyq_config* c, const void* q_proxy,
                                          int32_t n_proxy, int32_t n_proxy_ld, const void* k_src,
                                          int32_t ld, int32_t L, int32_t* idx_out, int32_t* k_out,
                                          void* ws, size_t ws_bytes, hyq_stream_t s) {
  hyq_status st = hyq_config_check(c);
  if (st != HYQ_OK) return st;
  if (!k_out) return HYQ_ERR_INVALID_ARG;
  if (L < 0 || L > c->capacity) return HYQ_ERR_CAPACITY;
  if (ld < L || ld < 1 || n_proxy < 0 || n_proxy_ld < n_proxy) return HYQ_ERR_INVALID_ARG;
  int32_t P = L - c->window > 0 ? L - c->window : 0;
  int32_t k = hyq_vl_count(c, P);
  *k_out = k;
  if (k == 0) return HYQ_OK;
  if (!q_proxy || !k_src || !idx_out || !aligned(k_src, 16) || !aligned(q_proxy, 16))
    return HYQ_ERR_INVALID_ARG;
  if (n_proxy < 1) return HYQ_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, kAlign) || ws_bytes < hyq_select_ws_bytes(c, L)) return HYQ_ERR_WORKSPACE;
  if (c->vl_mode == HYQ_VL_PER_QUERY_HEAD)
    return from_cuda(hyq_launch_select_heads(c, q_proxy, n_proxy, n_proxy_ld, k_src, ld, L, nullptr,
                                             hyq_vl_count_head(c, P), idx_out, k, ws, s));
  return from_cuda(hyq_launch_select(c, q_proxy, n_proxy, n_proxy_ld, k_src, ld, L, idx_out, k, ws, s));
}

extern "C" hyq_status hyq_select_vertical_heads(const hyq_config* c, const void* q_proxy, int32_t n_proxy,
                                                int32_t n_proxy_ld, const void* k_src, int32_t ld, int32_t L,
                                                int32_t* idx_heads_out, int32_t* idx_out, int32_t* k_out,
                                                int32_t* ku_out, void* ws, size_t ws_bytes, hyq_stream_t s) {
  hyq_status st = hyq_config_check(c);
  if (st != HYQ_OK) return st;
  if (c->vl_mode != HYQ_VL_PER_QUERY_HEAD || !k_out || !ku_out) return HYQ_ERR_INVALID_ARG;
  if (L < 0 || L > c->capacity) return HYQ_ERR_CAPACITY;
  if (ld < L || ld < 1 || n_proxy < 0 || n_proxy_ld < n_proxy) return HYQ_ERR_INVALID_ARG;
  const int32_t P = L - c->window > 0 ? L - c->window : 0;
  const int32_t k1 = hyq_vl_count_head(c, P), ku = hyq_vl_count(c, P);
  *k_out = k1;
  *ku_out = ku;
  if (k1 == 0) return HYQ_OK;
  if (!q_proxy || !k_src || !idx_out || !aligned(k_src, 16) || !aligned(q_proxy, 16)) return HYQ_ERR_INVALID_ARG;
  if (n_proxy < 1) return HYQ_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, kAlign) || ws_bytes < hyq_select_ws_bytes(c, L)) return HYQ_ERR_WORKSPACE;
  return from_cuda(hyq_launch_select_heads(c, q_proxy, n_proxy, n_proxy_ld, k_src, ld, L, idx_heads_out, k1,
                                           idx_out, ku, ws, s));
}

extern "C" hyq_status hyq_select_vertical_mass(const hyq_config* c, const void* q_proxy, int32_t n_proxy,
                                               int32_t n_proxy_ld, const void* k_src, int32_t ld, int32_t L,
                                               int32_t* idx_out, int32_t* k_out, void* ws, size_t ws_bytes,
                                               hyq_stream_t s) {
  hyq_status st = hyq_config_check(c);
  if (st != HYQ_OK) return st;
  if (!k_out) return HYQ_ERR_INVALID_ARG;
  if (L < 0 || L > c->capacity) return HYQ_ERR_CAPACITY;
  if (c->vl_mode != HYQ_VL_PER_KV_HEAD) return HYQ_ERR_UNSUPPORTED;
  if (ld < L || ld < 1 || n_proxy < 0 || n_proxy_ld < n_proxy || n_proxy > c->period) return HYQ_ERR_INVALID_ARG;
  int32_t P = L - c->window > 0 ? L - c->window : 0;
  int32_t k = hyq_vl_count(c, P);
  *k_out = k;
  if (k == 0) return HYQ_OK;
  if (!q_proxy || !k_src || !idx_out || !aligned(k_src, 16) || !aligned(q_proxy, 16))
    return HYQ_ERR_INVALID_ARG;
  if (n_proxy < 1) return HYQ_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, kAlign) || ws_bytes < hyq_select_mass_ws_bytes(c, L)) return HYQ_ERR_WORKSPACE;
  return from_cuda(hyq_launch_select_mass(c, q_proxy, n_proxy, n_proxy_ld, k_src, ld, L, idx_out, k, ws, s));
}

extern "C" hyq_status hyq_rebuild(const hyq_config* c, const void* k_src, const void* v_src,
                                  int32_t ld, int32_t L, const int32_t* idx, int32_t k,
                                  const hyq_layout* l, hyq_stream_t s) {
  hyq_status st = hyq_config_check(c);
  if (st != HYQ_OK) return st;
  if (!layout_ok(l)) return HYQ_ERR_INVALID_ARG;
  if (L < 0 || L > c->capacity) return HYQ_ERR_CAPACITY;
  if (ld < L || ld < 1) return HYQ_ERR_INVALID_ARG;
  int32_t P = L - c->window > 0 ? L - c->window : 0;
  if (k < 0 || k > P) return HYQ_ERR_INVALID_ARG;
  if (k > hyq_cap_vl(c)) return HYQ_ERR_CAPACITY;
  if (L - P > hyq_cap_tail(c)) return HYQ_ERR_CAPACITY;
  if (L > 0 && (!k_src || !v_src || !aligned(k_src, 16) || !aligned(v_src, 16)))
    return HYQ_ERR_INVALID_ARG;
  if (k > 0 && !idx) return HYQ_ERR_INVALID_ARG;
  return from_cuda(hyq_launch_rebuild(c, k_src, v_src, ld, L, idx, k, l, s));
}

extern "C" hyq_status hyq_decode_append(const hyq_config* c, const void* q, const void* k_new,
                                        const void* v_new, const hyq_layout* l, void* k_src,
                                        void* v_src, int32_t ld, hyq_stream_t s) {
  hyq_status st = hyq_config_check(c);
  if (st != HYQ_OK) return st;
  if (!layout_ok(l) || !q || !k_new || !v_new) return HYQ_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_new, 16) || !aligned(v_new, 16)) return HYQ_ERR_INVALID_ARG;
  if ((k_src == nullptr) != (v_src == nullptr)) return HYQ_ERR_INVALID_ARG;
  if (k_src && (ld < 1 || !aligned(k_src, 16) || !aligned(v_src, 16))) return HYQ_ERR_INVALID_ARG;
  return from_cuda(hyq_launch_decode_append(c, q, k_new, v_new, l, k_src, v_src, ld, s));
}

extern "C" hyq_status hyq_decode_attention(const hyq_config* c, const void* q,
                                           const hyq_layout* l, void* out, int32_t len_hint,
                                           void* ws, size_t ws_bytes, hyq_stream_t s) {
  hyq_status st = hyq_config_check(c);
  if (st != HYQ_OK) return st;
  if (!layout_ok(l) || !q || !out || len_hint < 0) return HYQ_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16)) return HYQ_ERR_INVALID_ARG;
  if (len_hint == 0 || len_hint > c->capacity) len_hint = c->capacity;
  if (!ws || !aligned(ws, kAlign) || ws_bytes < hyq_decode_ws_bytes(c, len_hint))
    return HYQ_ERR_WORKSPACE;
  return from_cuda(hyq_launch_decode(c, q, l, out, len_hint, ws, s));
}

extern "C" hyq_status hyq_decode_step(const hyq_config* c, const void* q, const void* k_new,
                                      const void* v_new, const hyq_layout* l, void* k_src, void* v_src,
                                      int32_t ld, void* out, int32_t len_hint, void* ws, size_t ws_bytes,
                                      hyq_stream_t s) {
  return hyq_decode_step_prefetch(c, q, k_new, v_new, l, nullptr, k_src, v_src, ld, out, len_hint, ws, ws_bytes,
                                  s);
}

extern "C" hyq_status hyq_decode_step_prefetch(const hyq_config* c, const void* q, const void* k_new,
                                               const void* v_new, const hyq_layout* l, const hyq_layout* next,
                                               void* k_src, void* v_src, int32_t ld, void* out, int32_t len_hint,
                                               void* ws, size_t ws_bytes, hyq_stream_t s) {
  hyq_status st = hyq_config_check(c);
  if (st != HYQ_OK) return st;
  if (!layout_ok(l) || !q || !k_new || !v_new || !out || len_hint < 0) return HYQ_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(out, 16))
    return HYQ_ERR_INVALID_ARG;
  if ((k_src == nullptr) != (v_src == nullptr)) return HYQ_ERR_INVALID_ARG;
  if (k_src && (ld < 1 || !aligned(k_src, 16) || !aligned(v_src, 16))) return HYQ_ERR_INVALID_ARG;
  if (len_hint == 0 || len_hint > c->capacity) len_hint = c->capacity;
  if (next && !layout_ok(next)) return HYQ_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, kAlign) || ws_bytes < hyq_decode_ws_bytes(c, len_hint)) return HYQ_ERR_WORKSPACE;
  return from_cuda(hyq_launch_decode(c, q, l, out, len_hint, ws, s, k_new, v_new, k_src, v_src, ld, next));
}

static hyq_status prefill_call(const hyq_config* c, int32_t dtype, const void* q, int32_t ldq, const void* k,
                               const void* v, int32_t ldk, int32_t L, const int32_t* vl_idx, int32_t kvl,
                               void* out, int32_t* err, void* ws, size_t ws_bytes, hyq_stream_t s, bool band) {
  hyq_status st = hyq_config_check(c);
  if (st != HYQ_OK) return st;
  if (dtype != HYQ_PREFILL_INT8 && dtype != HYQ_PREFILL_FP8 && dtype != HYQ_PREFILL_FP4) return HYQ_ERR_INVALID_ARG;
  if (L < 0 || L > c->capacity) return HYQ_ERR_CAPACITY;
  if (L == 0) return HYQ_OK;
  if (ldq < L || ldk < L) return HYQ_ERR_INVALID_ARG;
  int32_t P = L - c->window > 0 ? L - c->window : 0;
  if (kvl < 0 || kvl > P || (kvl > 0 && !vl_idx)) return HYQ_ERR_INVALID_ARG;
  if (!q || !k || !v || !out) return HYQ_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16)) return HYQ_ERR_INVALID_ARG;
  if ((L + 127) / 128 > 65535) return HYQ_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, kAlign) || ws_bytes < hyq_prefill_ws_bytes(c, dtype, L, kvl, band))
    return HYQ_ERR_WORKSPACE;
  return from_cuda(hyq_launch_prefill(c, dtype, q, ldq, k, v, ldk, L, vl_idx, kvl, out, ws, err, s, band));
}

extern "C" hyq_status hyq_prefill_attention(const hyq_config* c, int32_t dtype, const void* q,
                                            int32_t ldq, const void* k, const void* v, int32_t ldk,
                                            int32_t L, const int32_t* vl_idx, int32_t kvl, void* out,
                                            int32_t* err, void* ws, size_t ws_bytes, hyq_stream_t s) {
  return prefill_call(c, dtype, q, ldq, k, v, ldk, L, vl_idx, kvl, out, err, ws, ws_bytes, s, false);
}

extern "C" hyq_status hyq_prefill_attention_band(const hyq_config* c, int32_t dtype, const void* q,
                                                 int32_t ldq, const void* k, const void* v, int32_t ldk,
                                                 int32_t L, const int32_t* vl_idx, int32_t kvl, void* out,
                                                 int32_t* err, void* ws, size_t ws_bytes, hyq_stream_t s) {
  return prefill_call(c, dtype, q, ldq, k, v, ldk, L, vl_idx, kvl, out, err, ws, ws_bytes, s, true);
}

extern "C" hyq_status hyq_read_device_error(const int32_t* err_dev, int32_t* err_host,
                                            hyq_stream_t s) {
  if (!err_dev || !err_host) return HYQ_ERR_INVALID_ARG;
  cudaError_t e = cudaMemcpyAsync(err_host, err_dev, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return HYQ_ERR_CUDA;
  return *err_host ? HYQ_ERR_DEVICE : HYQ_OK;
}
