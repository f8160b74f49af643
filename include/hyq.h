/*
 * hyq.h -- C ABI of libhyq: hybrid-precision (4-bit + BF16) KV-cache attention
 * for one NVIDIA GB300 GPU (sm_103a).
 *
 * The method is the one of "HyQuant: Hybrid-Precision Quantization for LLM
 * Attention": per layer and KV head, the key/value positions are split into a
 * small set of vertical-line positions and a recent window, kept in BF16, and
 * the remaining majority, stored as asymmetric low-bit codes (§4.1 Eq. 1-3,
 * §4.3 Eq. 8): 4-bit keys and values by default, 8-bit keys and/or values
 * when hyq_config.bits_k / bits_v ask for them.  Decode attention
 * dequantises the quantised rows inside one online-softmax pass (§4.3 Eq. 9,
 * Appendix A.3 Algorithm 3).
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - Pointers named "device" point to GPU global memory owned by the caller;
 *    "host" pointers to CPU memory.  The library never allocates memory and
 *    never synchronises the stream (except hyq_read_device_error).
 *  - All calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).
 *  - Arguments are validated on the host first; an invalid call returns an
 *    error status before anything is launched and leaves all buffers as they
 *    were.  Errors that only the GPU can see (a value out of range, a count
 *    over capacity) set bits in a device error word instead (HYQ_DEVERR_*),
 *    which the caller reads with hyq_read_device_error; the kernels never
 *    trap and never wait on another block.
 *  - BF16 tensors are passed as `void*` and hold IEEE bfloat16 values;
 *    FP16 metadata is IEEE binary16.  All arrays are row-major and densely
 *    packed unless a leading dimension is given.
 *  - Only head_dim = 128, group = 32 and 1 <= HQ/HKV <= 8 are supported.
 */
#ifndef HYQ_H
#define HYQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *hyq_stream_t; /* same type as cudaStream_t */

typedef enum {
  HYQ_OK = 0,
  HYQ_ERR_INVALID_ARG = 1, /* null pointer, bad size or unsupported shape   */
  HYQ_ERR_UNSUPPORTED = 2, /* valid request this build does not implement   */
  HYQ_ERR_WORKSPACE = 3,   /* workspace null, misaligned or too small        */
  HYQ_ERR_CAPACITY = 4,    /* a length exceeds what the layout was sized for */
  HYQ_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed           */
  HYQ_ERR_DEVICE = 6       /* the device error word is non-zero              */
} hyq_status;

/* Bits of the device error word (an int32 in device memory). */
#define HYQ_DEVERR_QUANT_RANGE 0x1 /* a group's scale or zero is not a finite FP16, or NaN input */
#define HYQ_DEVERR_COUNT 0x2       /* a device-side count exceeded the layout capacity */
#define HYQ_DEVERR_INDEX 0x4       /* an index list was not strictly ascending in range */
#define HYQ_DEVERR_SCORE 0x8       /* a selection score was NaN */
#define HYQ_DEVERR_TIMEOUT 0x10    /* a bounded wait inside a kernel gave up (a bulk copy or a
                                      tensor-core commit did not complete); the kernel stopped
                                      issuing work, drained what it had in flight and returned */

/* Shape and method parameters of one attention layer. */
typedef struct {
  int32_t batch;        /* B >= 1                                               */
  int32_t num_q_heads;  /* HQ                                                   */
  int32_t num_kv_heads; /* HKV; HQ % HKV == 0 and g = HQ / HKV in [1, 8]         */
  int32_t head_dim;     /* d; must be 128                                       */
  int32_t group;        /* G, elements per quantisation group along d; must be 32 */
  int32_t window;       /* W >= 0, BF16 window length (128 in the paper)        */
  int32_t period;       /* re-selection period and proxy-query count (64)      */
  int32_t rho_ppm;      /* vertical-line ratio rho in parts per million (5% = 50000) */
  int32_t capacity;     /* largest context length L the layout must hold        */
  int32_t bits_k;       /* B_K, key code width: 4 or 8 (0 means 4)              */
  int32_t bits_v;       /* B_V, value code width: 4 or 8 (0 means 4)            */
  int32_t vl_mode;      /* HYQ_VL_PER_KV_HEAD (0) or HYQ_VL_PER_QUERY_HEAD       */
} hyq_config;

/*
 * Vertical-line granularity (hyq_config.vl_mode).  The cache holds one
 * vertical-line list per (sequence, KV head) in both modes: a position is
 * kept in BF16, or in the quantised stream, for the whole KV head.
 *   HYQ_VL_PER_KV_HEAD     one set per KV head, scored with the proxies of
 *                          all g query heads of the group summed; k =
 *                          min(P, max(1, ceil(P rho))) positions.
 *   HYQ_VL_PER_QUERY_HEAD  Algorithm 1's output as written, one set of k
 *                          positions per query head (B x H_Q x k), each
 *                          scored with that head's own proxies; the list
 *                          stored per KV head is the union of its g query
 *                          heads' sets, filled up to min(P, g k) positions
 *                          with the largest group scores (the per-KV-head
 *                          score) among the others, ties to the lower
 *                          position, so that every query head's own set is
 *                          held in BF16 and the list length is the same for
 *                          every head.  hyq_vl_count gives that length.
 */
#define HYQ_VL_PER_KV_HEAD 0
#define HYQ_VL_PER_QUERY_HEAD 1

/*
 * Quantised stream format.  The quantised ("4-bit") stream of one (batch, KV
 * head) is an array of 16-row tiles of HYQ_QTILE_BYTES_BITS(B_K, B_V) bytes
 * each, tile i holding stream rows 16i..16i+15; four consecutive tiles form a
 * block of HYQ_QBLOCK_ROWS rows, the unit the stream is allocated in.  With
 * CK = 256 B_K and CV = 256 B_V (the code bytes of 16 rows) a tile is
 *
 *   [0,            CK)           K codes
 *   [CK,           CK+CV)        V codes
 *   [CK+CV,        CK+CV+256)    K metadata: 16 rows x 4 groups x FP16 scale and zero
 *   [CK+CV+256,    CK+CV+512)    V metadata: same values, another order
 *
 * (B_K = B_V = 4: 1024 + 1024 + 256 + 256 = HYQ_QTILE_BYTES.)
 *
 * Metadata order (byte offsets inside the 256-byte region, r = row 0..15,
 * q = group 0..3, each entry one FP16):
 *   K: scale of (r, q) at 16*r + 2*q, zero at 16*r + 8 + 2*q
 *      (a row's four scales, then its four zeros);
 *   V: scale of (r, q) at 16*(r/2) + 4*q + 2*(r%2), zero 128 bytes further
 *      (rows paired (2i, 2i+1): one FP16 pair per pair of rows and group).
 * The dequantised value of element e (group q = e/32) is c * s + z with c
 * the B_K- (K) or B_V-bit (V) code.
 *
 * Inside a 4-bit (1024-byte) code region the 16 x 128 codes are ordered for the
 * register fragments of 16x16 tensor-core tiles: byte offset
 *   512*(u/4) + 16*lane + 4*(u%4)          (u = 0..7, lane = 0..31)
 * holds a 32-bit word whose nibble n (bits 4n..4n+3, n = 0..7) is the code
 * of, with g = lane/4, t = lane%4, a = n&1, b = (n>>1)&1, c = n>>2,
 *   K: row g + 8a,          element 8*(t + 4*(u/2)) + 4*(u%2) + 2b + c
 *   V: row 2t + 8b + c,     element 32*(u/2) + 4g + 2*(u%2) + a
 * An 8-bit code region (2048 bytes) holds one code per byte: byte offset
 *   512*(u/4) + 16*lane + 4*(u%4) + j      (u = 0..15, lane = 0..31, j = 0..3)
 * is the code of
 *   K: row g + 8*(u%2),          element 16*(u/2) + 4t + (0, 2, 1, 3)[j]
 *   V: row 2t + (0, 8, 1, 9)[j],  element 32*(u/4) + 4g + 2*((u/2)%2) + u%2
 * (the V output elements of m-tile u/2 are those of the 4-bit order).
 * Rows past the stream length inside the last block have zero codes and
 * zero metadata.
 */
#define HYQ_QBLOCK_ROWS 64
#define HYQ_QTILE_ROWS 16
#define HYQ_QTILE_BYTES_BITS(bk, bv) (256 * ((bk) + (bv)) + 512)
#define HYQ_QBLOCK_BYTES_BITS(bk, bv) (4 * HYQ_QTILE_BYTES_BITS(bk, bv))
#define HYQ_QBLOCK_BYTES 10240 /* B_K = B_V = 4 */
#define HYQ_QTILE_BYTES 2560   /* B_K = B_V = 4 */

/*
 * Device buffers of one layer's hybrid cache (§4.3 Eq. 8, Algorithm 4's four
 * buffers, with the staging buffer and the window held as one BF16 tail).
 * Sizes in bytes come from hyq_layout_sizes(); all pointers are device
 * pointers, 256-byte aligned.
 *
 *   qblocks  [B][HKV][nblk][HYQ_QBLOCK_BYTES_BITS(B_K, B_V)]  quantised stream: row r is
 *            position r, for every position r < NQ that has left the BF16 tail;
 *            the rows of vertical-line positions keep their codes but their
 *            four key steps are FP16 NaN (decode leaves those rows out; their
 *            values are the BF16 vertical-line rows)
 *   vl_k/v   bf16 [B][HKV][cap_vl][128]  vertical-line rows, ascending position
 *   vl_idx   int32 [B][HKV][cap_vl]      their positions
 *   tail_k/v bf16 [B][HKV][cap_tail][128] positions [P, L) in order
 *   q_ring   bf16 [B][HQ][period][128]   the `period` most recent queries
 *   counts   int32 [B][HYQ_COUNTS]       see HYQ_CNT_*
 *   err      int32 [1]                    device error word
 * with nblk = ceil(capacity / 64), cap_vl = vertical-line count at
 * capacity, cap_tail = window + period.
 */
typedef struct {
  uint8_t *qblocks;
  void *vl_k;
  void *vl_v;
  int32_t *vl_idx;
  void *tail_k;
  void *tail_v;
  void *q_ring;
  int32_t *counts;
  int32_t *err;
} hyq_layout;

#define HYQ_COUNTS 8
#define HYQ_CNT_NQ 0       /* rows in the 4-bit stream (positions 0..NQ-1) */
#define HYQ_CNT_NVL 1      /* vertical-line rows                           */
#define HYQ_CNT_NTAIL 2    /* BF16 tail rows                               */
#define HYQ_CNT_LEN 3      /* context length L = NQ + NTAIL                */
#define HYQ_CNT_RING_N 4   /* valid entries in q_ring (<= period)          */
#define HYQ_CNT_RING_POS 5 /* next q_ring slot                             */

#define HYQ_LAYOUT_FIELDS 9 /* qblocks vl_k vl_v vl_idx tail_k tail_v q_ring counts err */

#define HYQ_OP_SELECT 1
#define HYQ_OP_DECODE 2
#define HYQ_OP_PREFILL 3
#define HYQ_OP_SELECT_MASS 4
#define HYQ_OP_PREFILL_BAND 5

#define HYQ_PREFILL_INT8 1
#define HYQ_PREFILL_FP8 2
#define HYQ_PREFILL_FP4 3

/* Human-readable name of a status. */
const char *hyq_status_string(hyq_status s);

/* Validate a config; HYQ_OK when every entry point accepts it. */
hyq_status hyq_config_check(const hyq_config *cfg);

/* Length of the per-KV-head vertical-line list for a prefix of P positions:
 * k = min(P, max(1, ceil(P * rho))) (Algorithm 1), and 0 when P <= 0 or
 * rho = 0; with vl_mode = HYQ_VL_PER_QUERY_HEAD, min(P, g k).
 * Returns -1 for a null config. */
int32_t hyq_vl_count(const hyq_config *cfg, int32_t P);

/* Bytes of each layout field, in the order of HYQ_LAYOUT_FIELDS
 * (out[HYQ_LAYOUT_FIELDS], host). */
hyq_status hyq_layout_sizes(const hyq_config *cfg, size_t *out);

/* Workspace bytes an operation needs (HYQ_OP_*); 0 on an invalid config.
 * A workspace must be zero-filled before its first use; the kernels leave it
 * ready for the next call.  `len_hint` is the largest context length the
 * call will see (0 = capacity). */
size_t hyq_workspace_size(const hyq_config *cfg, int op, int32_t len_hint);

/* Zero the counters and the error word of a layout (the empty cache). */
hyq_status hyq_layout_reset(const hyq_config *cfg, const hyq_layout *lay, hyq_stream_t stream);

/*
 * Quant_B(.; G) of Algorithm 4 (Appendix A.4) and the low-bit cache of §4.3
 * Eq. 8: quantise n_rows new rows per (batch, KV head) of K and V and append
 * them to the quantised stream after its current NQ rows.
 *   k_rows, v_rows  device bf16 [B][HKV][n_rows][128]
 * Per group of 32 elements along head_dim, with mn/mx the group min/max and
 * qmax = 2^B - 1 (B = bits_k for K, bits_v for V: 15 or 255):
 *   s = FP16 value of (mx - mn) / qmax (exact quotient) rounded toward +inf,
 *   z = FP16 value of mn rounded to nearest even,
 *   c = the integer in [0, qmax] nearest to (x - z) / s, ties to even (the
 *       grid point z + c s nearest to x; c = 0 when s = 0), decided exactly.
 * A group with a non-finite s or z gets zero codes, s = z = 0 and sets
 * HYQ_DEVERR_QUANT_RANGE.  Rows that would pass the capacity are dropped and
 * set HYQ_DEVERR_COUNT.  Updates NQ and LEN.
 */
hyq_status hyq_quantize_append(const hyq_config *cfg, const void *k_rows, const void *v_rows,
                               int32_t n_rows, const hyq_layout *lay, hyq_stream_t stream);

/*
 * Frozen-mode maintenance (Algorithm 4 as written, Appendix A.4: the
 * vertical-line set is fixed at freeze and only positions that leave the
 * window are quantised).  For every sequence b, the oldest
 * m = max(0, NTAIL - W) tail rows (positions [L - NTAIL, L - W)) are
 * quantised exactly as hyq_quantize_append does and appended to the 4-bit
 * stream after its NQ rows, and the last W tail rows move to the front of the
 * tail: NQ += m, NTAIL -= m, LEN, the vertical-line rows and the proxy ring
 * unchanged.  The layout afterwards is that of hyq_rebuild at LEN with the
 * same index list.  A sequence whose counters are out of range or whose
 * stream has no room for the m rows is left unchanged and sets
 * HYQ_DEVERR_COUNT.  Three launches, no workspace.
 */
hyq_status hyq_age_tail(const hyq_config *cfg, const hyq_layout *lay, hyq_stream_t stream);

/*
 * Vertical-line token identification, Eq. 4-5 and Algorithm 1 (Appendix A.1).
 *   q_proxy  device bf16 [B][HQ][n_proxy_ld][128]; the first n_proxy query
 *            rows of each head are used (order does not matter)
 *   k_src    device bf16 [B][HKV][ld][128], the BF16 keys, ld >= L
 *   idx_out  device int32 [B][HKV][k]: positions, strictly ascending
 *   k_out    host int32: k = hyq_vl_count(cfg, max(0, L - window))
 * Per KV head: u = sum over the n_proxy proxy queries and the g query heads
 * of the group; S(j) = u . k_j for j < P = max(0, L - W) in float32; the k
 * positions with the largest S, ties to the lower position.
 * Workspace: hyq_workspace_size(cfg, HYQ_OP_SELECT, L).
 */
hyq_status hyq_select_vertical(const hyq_config *cfg, const void *q_proxy, int32_t n_proxy,
                               int32_t n_proxy_ld, const void *k_src, int32_t ld, int32_t L,
                               int32_t *idx_out, int32_t *k_out, void *ws, size_t ws_bytes,
                               hyq_stream_t stream);

/*
 * Algorithm 1 per query head (Appendix A.1, output B x H_Q x k), for a config
 * with vl_mode = HYQ_VL_PER_QUERY_HEAD (any other config: HYQ_ERR_INVALID_ARG).
 *   q_proxy, n_proxy, k_src, ld, L  as for hyq_select_vertical
 *   idx_heads_out  device int32 [B][HQ][k] or NULL: each query head's set,
 *                  strictly ascending
 *   idx_out        device int32 [B][HKV][ku]: the stored list, strictly
 *                  ascending (the union of the group's sets filled up to ku
 *                  by the group score, see HYQ_VL_PER_QUERY_HEAD)
 *   k_out, ku_out  host int32: k = min(P, max(1, ceil(P rho))) and
 *                  ku = hyq_vl_count(cfg, P) = min(P, g k)
 * Query head h scores S_h(j) = u_h . k_j (u_h the sum of its n_proxy proxy
 * queries, k_j the key of h's KV head) and keeps its k largest, ties to the
 * lower position; the group score is hyq_select_vertical's.  Both in
 * float32.  hyq_select_vertical on such a config computes the same idx_out.
 * Workspace: hyq_workspace_size(cfg, HYQ_OP_SELECT, L).  Six launches.
 */
hyq_status hyq_select_vertical_heads(const hyq_config *cfg, const void *q_proxy, int32_t n_proxy,
                                     int32_t n_proxy_ld, const void *k_src, int32_t ld, int32_t L,
                                     int32_t *idx_heads_out, int32_t *idx_out, int32_t *k_out,
                                     int32_t *ku_out, void *ws, size_t ws_bytes, hyq_stream_t stream);

/*
 * Vertical-line identification with the score of Eq. 4 (§4.1): the
 * accumulated column mass of the attention probabilities instead of
 * Algorithm 1's summed logits.  Same arguments and output as
 * hyq_select_vertical, and n_proxy <= cfg->period.  Per KV head, with the
 * rows r = (query head i of the group, proxy t) and alpha = 1/sqrt(d):
 *   a_rj = softmax over the L keys j < L of alpha q_r . k_j
 *   S(j) = sum_r a_rj for j < P = max(0, L - W)
 * then the k positions with the largest S, ties to the lower position.
 * Evaluated in float32 from exact BF16 products on the tensor cores: per
 * row the maximum m of t = (q_r . k_j) fl(alpha log2 e) and the sum l of
 * 2^(t - m), over at most 32 key ranges merged once, then
 * S(j) = sum_r 2^(t - m) / l; a NaN score sets HYQ_DEVERR_SCORE in the
 * workspace's error word.  k_src and q_proxy must be 16-byte aligned (they
 * are read through TMA tensor maps).
 * Per KV head only: a config with vl_mode = HYQ_VL_PER_QUERY_HEAD returns
 * HYQ_ERR_UNSUPPORTED.
 * Workspace: hyq_workspace_size(cfg, HYQ_OP_SELECT_MASS, L).  Three launches
 * when a KV group's proxy rows (g n_proxy) fit one group of 256, four beyond.
 */
hyq_status hyq_select_vertical_mass(const hyq_config *cfg, const void *q_proxy, int32_t n_proxy,
                                    int32_t n_proxy_ld, const void *k_src, int32_t ld, int32_t L,
                                    int32_t *idx_out, int32_t *k_out, void *ws, size_t ws_bytes,
                                    hyq_stream_t stream);

/*
 * Build a layer's hybrid cache for context length L (Algorithm 4, with the
 * vertical-line set re-chosen): the 4-bit stream holds the positions [0, P),
 * row = position, quantised as in hyq_quantize_append, those of idx marked
 * (NaN key steps); the vertical-line buffers hold the BF16 rows of idx; the
 * tail holds [P, L).  Rows already in the stream (positions below its NQ)
 * are kept: only [NQ, P) is quantised, and the marks move from the previous
 * vertical-line set to idx (a position leaving the set gets its key steps
 * back from its BF16 row), so a re-selection costs O(64 + k), not O(P).
 * The stream must therefore hold the same sequence as k_src: reset the
 * layout (hyq_layout_reset) before building it for another one.
 *   k_src, v_src  device bf16 [B][HKV][ld][128]
 *   idx           device int32 [B][HKV][k], strictly ascending in [0, P)
 * Sets NQ = P, NVL = k, NTAIL = L - P, LEN = L.  Leaves q_ring alone.
 * An idx list that is not strictly ascending within [0, P) sets
 * HYQ_DEVERR_INDEX (the output is then unspecified but in bounds).
 */
hyq_status hyq_rebuild(const hyq_config *cfg, const void *k_src, const void *v_src, int32_t ld,
                       int32_t L, const int32_t *idx, int32_t k, const hyq_layout *lay,
                       hyq_stream_t stream);

/*
 * One decode step's bookkeeping (Algorithm 3 inputs, §5.5 query buffer):
 * append this step's key/value row to the BF16 tail, store the query in the
 * proxy ring, and (when k_src/v_src are non-null) write the row into the
 * caller's BF16 cache at position LEN.  Updates NTAIL, LEN, RING_N, RING_POS.
 *   q        device bf16 [B][HQ][128]
 *   k_new    device bf16 [B][HKV][128];  v_new likewise
 *   k_src    device bf16 [B][HKV][ld][128] or NULL;  v_src likewise
 * A full tail (NTAIL = window + period) or LEN >= ld drops the row and sets
 * HYQ_DEVERR_COUNT.
 */
hyq_status hyq_decode_append(const hyq_config *cfg, const void *q, const void *k_new,
                             const void *v_new, const hyq_layout *lay, void *k_src,
                             void *v_src, int32_t ld, hyq_stream_t stream);

/*
 * Hybrid-precision decode attention, §4.3 Eq. 8-9 and Algorithm 3 (Appendix
 * A.3): for every query head h (KV head h / g)
 *   out_h = sum_j exp(a q_h.k~_j - M) v~_j / sum_j exp(a q_h.k~_j - M),
 * a = 1/sqrt(128), over the LEN positions of the layout, with k~, v~ the
 * dequantised rows of the quantised stream (c*s + z, B_K- and B_V-bit codes)
 * and the BF16 vertical-line and tail rows.
 * The quantised stream is split along the sequence across thread blocks, the g
 * query heads of a KV head are processed together, and the split partials
 * are merged by log-sum-exp rescaling in the same launch.
 *   q    device bf16 [B][HQ][128]
 *   out  device bf16 [B][HQ][128] (zeros when LEN = 0)
 *   len_hint  an upper bound of the current context lengths, used only to
 *        size the launch (0 = capacity)
 * Workspace: hyq_workspace_size(cfg, HYQ_OP_DECODE, len_hint), zero-filled
 * before first use; one workspace must not be used by two calls at once.
 */
hyq_status hyq_decode_attention(const hyq_config *cfg, const void *q, const hyq_layout *lay,
                                void *out, int32_t len_hint, void *ws, size_t ws_bytes,
                                hyq_stream_t stream);

/*
 * Hybrid-precision prefill attention, §4.2 Eq. 6-7 and Algorithm 2 (Appendix
 * A.2), causal, for every query row i < L and query head h (KV head h / g):
 *   out_{h,i} = softmax_j(x_j) . v_j over j <= i, a = 1/sqrt(128), where for
 *   j in the full-precision set (the vertical lines vl_idx and the last W
 *   positions [P, L), P = max(0, L - W)) x_j = a q_i . k_j and v_j are the BF16
 *   rows, and for the other positions of [0, P) (the quantised prefix)
 *   x_j = a q^_i . k^_j and v_j = v^_j, with
 *   - the quantised-prefix positions taken in ascending order and cut into
 *     tiles of 64 (the last one may be shorter); per tile one scale for K
 *     and one for V: s = fl32(max|x| / c) over the tile, c = 127 (INT8),
 *     448 (FP8 e4m3) or 6 (FP4 e2m1);
 *   - one scale for Q per block of 128 consecutive rows of one head
 *     (rows 128m .. 128m+127, those < L);
 *   - the code of x is the grid value nearest to the exact quotient x / s,
 *     ties to the even code: INT8 the integers -127..127, FP8 the e4m3
 *     values (saturating at +-448), FP4 the e2m1 values 0, 0.5, 1, 1.5, 2,
 *     3, 4, 6 and their negatives (saturating at +-6); x^ = code * s.
 *   dtype  HYQ_PREFILL_INT8, HYQ_PREFILL_FP8 or HYQ_PREFILL_FP4
 *   q      device bf16 [B][HQ][ldq][128]; rows 0..L-1 are used
 *   k, v   device bf16 [B][HKV][ldk][128]
 *   vl_idx device int32 [B][HKV][kvl], strictly ascending in [0, P)
 *          (e.g. from hyq_select_vertical); kvl may be 0
 *   out    device bf16 [B][HQ][L][128]
 *   err    device int32 [1] or NULL: HYQ_DEVERR_INDEX for an invalid vl_idx
 *          (the output is then unspecified), HYQ_DEVERR_TIMEOUT
 * The softmax probabilities enter the P.V product rounded to BF16 (the value
 * scale folded in); all products accumulate in float32.
 * Workspace: hyq_workspace_size(cfg, HYQ_OP_PREFILL, L) covers every call
 * with context length <= L and kvl <= hyq_vl_count(cfg, P); it needs no
 * zero fill.  L > capacity returns HYQ_ERR_CAPACITY.
 */
hyq_status hyq_prefill_attention(const hyq_config *cfg, int32_t dtype, const void *q, int32_t ldq,
                                 const void *k, const void *v, int32_t ldk, int32_t L,
                                 const int32_t *vl_idx, int32_t kvl, void *out, int32_t *err,
                                 void *ws, size_t ws_bytes, hyq_stream_t stream);

/*
 * Hybrid-precision prefill attention with the window taken per query (a
 * diagonal band) instead of as the last W positions: the reading of
 * Algorithm 2's window (Appendix A.2) in which every query keeps its own most
 * recent keys in full precision.  Query row i sees
 *   - the keys (i - W, i] as BF16 rows (its band),
 *   - the vertical lines at or before i - W as BF16 rows,
 *   - every other key at or before i - W from the quantised prefix,
 * where vl_idx, the quantised-prefix positions ([0, P) minus vl_idx), their
 * tiles, scales and codes, and the query scales are exactly those of
 * hyq_prefill_attention (for every row i - W <= P - 1, so no other key is
 * needed in quantised form).  The last row, and every row when W = 0, equal
 * hyq_prefill_attention's.  Arguments, layouts, error reporting and
 * asynchrony as hyq_prefill_attention.
 * Workspace: hyq_workspace_size(cfg, HYQ_OP_PREFILL_BAND, L) covers every
 * call with context length <= L and kvl <= hyq_vl_count(cfg, P); it holds
 * BF16 images of all L key and value rows in addition to the code images.
 */
hyq_status hyq_prefill_attention_band(const hyq_config *cfg, int32_t dtype, const void *q,
                                      int32_t ldq, const void *k, const void *v, int32_t ldk,
                                      int32_t L, const int32_t *vl_idx, int32_t kvl, void *out,
                                      int32_t *err, void *ws, size_t ws_bytes, hyq_stream_t stream);

/*
 * One decode step in one launch: hyq_decode_append followed by
 * hyq_decode_attention (§4.3 Eq. 8-9, Algorithm 3; §5.5 query buffer).  The
 * token's K/V row becomes the newest tail row (and row LEN of the caller's
 * BF16 cache when k_src/v_src are non-null), its query goes to the proxy
 * ring, the counters advance as in hyq_decode_append, and `out` is the
 * attention of q over the LEN + 1 positions, the new row included.
 * Arguments as in those two calls; len_hint bounds LEN + 1.  A full tail (or
 * LEN >= ld) sets HYQ_DEVERR_COUNT, leaves the layout unchanged and attends
 * over the LEN existing positions.  Workspace: hyq_workspace_size(cfg,
 * HYQ_OP_DECODE, len_hint), zero-filled before first use.
 */
hyq_status hyq_decode_step(const hyq_config *cfg, const void *q, const void *k_new,
                           const void *v_new, const hyq_layout *lay, void *k_src, void *v_src,
                           int32_t ld, void *out, int32_t len_hint, void *ws, size_t ws_bytes,
                           hyq_stream_t stream);

/*
 * hyq_decode_step that also warms L2 for the next decode call on the stream.
 * The paper has no counterpart: it overlaps the HBM reads of the next layer
 * with the end of this launch (the block reduction and split merge, when
 * most SMs and most of the HBM bandwidth are idle).
 *
 * Same arguments, result and layout updates as hyq_decode_step, plus
 *   next  the layout the next decode call will read (typically the next
 *         layer's), allocated for the same cfg; or NULL (no prefetch, the
 *         same launch as hyq_decode_step); may equal lay.
 * Once one warp of each block has read its tiles of lay, it issues L2 prefetches (bulk
 * prefetch hints, no data is written) for the share of next that the same
 * block index of a decode call with the same cfg and len_hint reads: its
 * 4-bit tiles and its vertical-line and tail rows, from next's counters at
 * the time (clamped to the capacities of cfg, so every address is inside
 * next's buffers).  Results never depend on next; a stale or concurrently
 * updated next only makes the hint less useful.  Errors as hyq_decode_step,
 * and HYQ_ERR_INVALID_ARG when next is non-NULL with a NULL buffer.
 */
hyq_status hyq_decode_step_prefetch(const hyq_config *cfg, const void *q, const void *k_new,
                                    const void *v_new, const hyq_layout *lay, const hyq_layout *next,
                                    void *k_src, void *v_src, int32_t ld, void *out, int32_t len_hint,
                                    void *ws, size_t ws_bytes, hyq_stream_t stream);

/*
 * Let hyq_decode_attention and hyq_decode_step launches overlap the kernel
 * launched before them on the same stream (programmatic dependent launch;
 * process-wide, off by default).  With it on, every such launch lets the next
 * launch on its stream start once the kernel before it has finished; it
 * reads the layer's layout (counters, 4-bit stream, vertical-line and tail
 * rows) before the preceding kernel has finished, and the query, the new
 * K/V row, the workspace and every output only after.  The caller guarantees
 * that the kernel launched immediately before each decode call on its stream
 * does not write that call's layout: true in a transformer decode step (that
 * kernel produces q, k, v) and between calls on different layers; false for
 * consecutive calls on the same layer, which must run with it off.
 * Returns HYQ_ERR_INVALID_ARG unless enable is 0 or 1.
 */
hyq_status hyq_set_decode_overlap(int32_t enable);

/*
 * Override how hyq_decode_attention splits and merges its work (process-
 * wide; for tuning and testing).  merge: 0 automatic (the default), 1 one
 * block per (batch, KV head) and no merge, 2 `splits` blocks (2..16) merged
 * inside a thread-block cluster, 3 `splits` blocks (1..1024) merged through
 * the workspace by the last block to finish.  The workspace size reported by
 * hyq_workspace_size follows the override.  Returns HYQ_ERR_INVALID_ARG for
 * values out of range and leaves the previous setting.
 */
hyq_status hyq_set_decode_plan(int32_t merge, int32_t splits);

/*
 * hyq_decode_attention without a caller-provided workspace.  The paper has
 * no counterpart; this exists for callers that cannot allocate device
 * memory: plugins and embedding runtimes that hand an attention op only its
 * inputs and outputs (no workspace argument, no allocator) and hot loops that
 * must not call cudaMalloc, which synchronises the device and can fail under
 * memory pressure.
 *
 * Same arguments, result and layout as hyq_decode_attention, minus `ws`.
 * The split partials and tickets live in a fixed library-owned device array
 * of HYQ_NOALLOC_SCRATCH_BYTES (4 MiB), present on every GPU that loads the
 * library until the process exits.  The call allocates nothing.
 *  - The first call on a device looks up that array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture.
 *  - A shape whose scratch need, hyq_workspace_size(cfg, HYQ_OP_DECODE,
 *    len_hint), exceeds HYQ_NOALLOC_SCRATCH_BYTES is rejected with
 *    HYQ_ERR_WORKSPACE before anything is launched.
 *  - Every call on a device shares the one array and each call re-zeroes the
 *    part that must start at zero (a memset on `stream` before the kernel);
 *    two calls that overlap on the GPU (other streams, other threads) race on
 *    it and give wrong results.
 *  - Because of that memset, hyq_set_decode_overlap has no effect on this
 *    entry point: its kernel is never launched as a programmatic dependent.
 */
#define HYQ_NOALLOC_SCRATCH_BYTES (4u << 20)
hyq_status hyq_decode_attention_noalloc(const hyq_config *cfg, const void *q, const hyq_layout *lay,
                                        void *out, int32_t len_hint, hyq_stream_t stream);

/*
 * Copy a device error word to the host (synchronises `stream`).
 *   err_dev  device int32 [1];  err_host  host int32 [1]
 * Returns HYQ_ERR_DEVICE when the word is non-zero, HYQ_OK otherwise.
 */
hyq_status hyq_read_device_error(const int32_t *err_dev, int32_t *err_host, hyq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* HYQ_H */
