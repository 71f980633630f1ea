/*
 * h3kv.h -- C ABI of libh3kv: the kvi8r rotated-int8 whole-sequence K/V store
 * and query-chunked attention over it, on one NVIDIA GB300 (sm_103a); the
 * exact bf16 comparison path; the kvf8s store (fp8 e4m3 in the kvi8s
 * layout) attended on the fp8 tensor path; and the kvfp4 store (NVFP4 K/V)
 * dequantised exactly to fp16 for the tensor cores.
 *
 * Source of the method: "H3 Streamed Blocks (exact low-VRAM, alpha)", Inputs
 * table (kv_store, q_chunk, kv_block rows), and "Low VRAM, low RAM: the
 * de-rope on a 16 GB card", section "The K/V store options" (kvi8r row and the
 * paragraph on why the rotation).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Layout: every tensor is contiguous, head-major [heads, seq, head_dim]
 *    with head_dim == 128; per-row scales are [heads, seq].  bf16 and fp16
 *    values are passed as their 16-bit patterns (uint16_t).
 *  - Memory: all tensor pointers are DEVICE pointers on the current CUDA
 *    device, 16-byte aligned, owned by the caller.  The library allocates no
 *    device memory and frees nothing.
 *  - Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).
 *    Calls are stream-ordered and asynchronous: they return after the launch.
 *  - Errors: argument checks run on the host before any launch and return
 *    H3KV_ERR_INVALID_ARG / H3KV_ERR_UNSUPPORTED with nothing launched.  A
 *    launch failure returns H3KV_ERR_CUDA.  Every wait inside the kernels is
 *    bounded; a wait that runs out records a device error word and the kernel
 *    returns early.  h3kv_sync_status() reports (and clears) that word.
 *  - Empty work (heads == 0 or a zero sequence length) returns H3KV_OK and
 *    launches nothing, except that attending a non-empty query set to an
 *    empty key set is H3KV_ERR_INVALID_ARG (the softmax has no terms).
 *  - Attention entry points take at most 65535 heads (one grid row per
 *    head); more is H3KV_ERR_INVALID_ARG.
 */
#ifndef H3KV_H
#define H3KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define H3KV_ABI_VERSION 9u
#define H3KV_HEAD_DIM 128
/* kv_block = 0 on the kvi8r path means this many tokens (the kv_block
 * default of the kv_store row). */
#define H3KV_DEFAULT_KV_BLOCK 16384
/* kv_block must be 0 or a multiple of this (the key tile of the kernels). */
#define H3KV_KV_TILE 128

typedef enum {
  H3KV_OK = 0,
  H3KV_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, bad size or chunk  */
  H3KV_ERR_UNSUPPORTED = 2,    /* head_dim != 128, or device is not sm_103   */
  H3KV_ERR_CUDA = 3,           /* a CUDA runtime call or launch failed       */
  H3KV_ERR_DEVICE_TIMEOUT = 4  /* a bounded in-kernel wait ran out           */
} h3kv_status;

/* The kvi8r store: for K and for V, int8 codes [heads, seq, 128] and fp16
 * scales.  The codes are the rows of K (or V) rotated into the orthonormal
 * Sylvester-Hadamard basis H (x' = x H, H the order-128 Hadamard matrix /
 * sqrt(128)), quantised per scale group G of consecutive rotated values as
 *   s = fp16_rne(max_{j in G} |x'_j| / 127)   (saturated at 65504),
 *   c_j = clamp(rne(x'_j / s), -127, 127),   c = 0 where s == 0.
 * Dequantisation is c * s.  scale_group selects the group:
 *   0 or 128: one scale per (head, token) row (the kv_store row of the H3
 *             Streamed Blocks Inputs table); scales are [heads, seq];
 *   32:       one scale per 32 values (the "per-32-value scale variant of
 *             kvi8r" of the Low VRAM write-up's roadmap); scales are
 *             [heads, seq, 4].
 * All four buffers are caller-owned memory (device memory, or host memory
 * the GPU can address -- see h3kv_attend_staged). */
typedef struct {
  int8_t *k_codes;
  int8_t *v_codes;
  uint16_t *k_scales; /* fp16 bit patterns */
  uint16_t *v_scales; /* fp16 bit patterns */
  int32_t heads;
  int64_t seq;
  int32_t head_dim;    /* must be 128 */
  int32_t scale_group; /* 0 or 128 (per row) or 32 */
} h3kv_store;

/* Version of this ABI (H3KV_ABI_VERSION). */
uint32_t h3kv_abi_version(void);

/* Bytes of device memory a per-row-scale store of this shape occupies in
 * total (codes and scales of K and V): 2 * heads * seq * (head_dim + 2); a
 * scale_group 32 store holds 6 more bytes per row and tensor.  Returns 0 for
 * invalid shapes. */
size_t h3kv_store_bytes(int32_t heads, int64_t seq, int32_t head_dim);

/* Build the kvi8r store from bf16 K and V [heads, seq, 128] (kv_store row of
 * the H3 Streamed Blocks Inputs table: rotate by the fixed Hadamard basis,
 * one fp16 absmax scale per token per head, int8 codes).  `out` describes the
 * destination buffers and must match heads/seq/head_dim.  K and V are read
 * once; codes and scales are written once.  K and V may be device memory or
 * pinned host memory that the GPU addresses (on a Grace-Blackwell node the
 * kernel reads them over NVLink-C2C), so the caller's K/V need never be
 * copied into HBM; the store is the same bit for bit. */
h3kv_status h3kv_build_store(const uint16_t *K, const uint16_t *V, int32_t heads, int64_t seq,
                             int32_t head_dim, const h3kv_store *out, void *stream);

/* kvi8r attention (kv_store row): O = softmax(q' K'^T * softmax_scale) V' H^T
 * where q' = Q H rounded to fp16, K' and V' are the dequantised store
 * (int8 -> fp16 cast times the fp16 scale), the softmax runs over all
 * store->seq keys (non-causal), in kv_block-token blocks combined by their
 * log-sum-exp, and the output is un-rotated once.
 *   Q: bf16 [store->heads, q_seq, 128].  O: fp32 [store->heads, q_seq, 128].
 *   q_chunk >= 1: query tokens per kernel launch (the q_chunk input).  The
 *     output is bit-identical for every q_chunk ("exact at any value").
 *   kv_block: 0 (= 16384) or a positive multiple of 128.
 *   softmax_scale <= 0 selects 1/sqrt(128). */
h3kv_status h3kv_attend(const uint16_t *Q, int64_t q_seq, const h3kv_store *store, int32_t q_chunk,
                        int32_t kv_block, float softmax_scale, float *O, void *stream);

/* The exact store (the "bf16 (exact)" kv_store option): plain softmax
 * attention on bf16 K and V, O = softmax(Q K^T * softmax_scale) V, with P
 * rounded to bf16 for the second product and fp32 accumulation.
 *   Q: bf16 [heads, q_seq, 128]; K, V: bf16 [heads, kv_seq, 128];
 *   O: fp32 [heads, q_seq, 128].
 *   q_chunk >= 1 as above (bit-identical for every value).
 *   kv_block: 0 (= one block over all keys) or a positive multiple of 128:
 *     keys are attended in blocks combined by their log-sum-exp (the kv_block
 *     input).
 *   softmax_scale <= 0 selects 1/sqrt(128). */
h3kv_status h3kv_attend_exact(const uint16_t *Q, int64_t q_seq, const uint16_t *K, const uint16_t *V,
                              int32_t heads, int64_t kv_seq, int32_t head_dim, int32_t q_chunk,
                              int32_t kv_block, float softmax_scale, float *O, void *stream);

/* Device bytes of the staging buffer h3kv_attend_staged needs: one kv_block
 * of codes and scales of K and V for every head, 2 * heads * kv_block * 130
 * (kv_block = 0 means 16384).  Returns 0 for invalid arguments. */
size_t h3kv_staging_bytes(int32_t heads, int32_t kv_block);

/* kvi8r attention over a store that lives outside HBM -- e.g. in pinned
 * Grace memory -- staged through HBM one kv_block at a time: the "host-staged
 * K/V design" the kv_block row of the H3 Streamed Blocks Inputs table keeps
 * the blockwise combine for.  For each block (in order) the block's codes and
 * scales of every head are copied into `staging` (device memory,
 * >= h3kv_staging_bytes(store->heads, kv_block)) and every query chunk
 * attends over it; the log-sum-exp combine across blocks is carried by
 * `state` (device fp32 [store->heads, q_seq, 2]: running max and sum per
 * query row) with O itself as the running un-normalised output.  The result
 * is bit-identical to h3kv_attend on the same store, q_chunk and kv_block.
 * Arguments otherwise as h3kv_attend; `store` may point to device, managed
 * or pinned (page-locked) host memory, and must have per-row scales
 * (scale_group 0 or 128; H3KV_ERR_UNSUPPORTED otherwise).  A store buffer in
 * pageable host memory is refused (H3KV_ERR_INVALID_ARG) before any work:
 * copies from pageable memory take its bytes when they are issued, not in
 * stream order, so a store built into it by earlier work still queued on
 * the GPU would be read before it is written.  The library allocates
 * nothing:
 * staging and state are caller-owned scratch, reused by each call, so calls
 * that overlap on the GPU must not share them.
 * With staging_bytes >= round_up(h3kv_staging_bytes(...), 256) +
 * h3kv_staging_bytes(...), two blocks are staged: the copy of block b + 1
 * runs on a second stream (created for the call) while block b is attended.
 * With less, each block's copy runs on `stream` between the blocks' launches.
 * Within a block, the launches of successive query chunks follow each other
 * as in h3kv_attend. */
h3kv_status h3kv_attend_staged(const uint16_t *Q, int64_t q_seq, const h3kv_store *store, int32_t q_chunk,
                               int32_t kv_block, float softmax_scale, float *O, void *staging,
                               size_t staging_bytes, float *state, void *stream);

/* Device scratch bytes h3kv_attend_hostio needs: two query chunks of Q
 * (bf16) and two of O (fp32) for every head, plus 256 bytes for the two
 * buffers' ready words: 2 * heads * q_chunk * 128 * 6 + 256.  Returns 0 for
 * invalid arguments. */
size_t h3kv_hostio_scratch_bytes(int32_t heads, int32_t q_chunk);

/* h3kv_attend with Q and O in host memory (pinned for asynchronous copies),
 * streamed through HBM one query chunk at a time -- the q_chunk input's way
 * of bounding the device transient.  The rows of chunk c are copied in, attended over
 * the (device-resident) store, and copied back.  The copies of other chunks
 * run on a second stream that the library creates for the call, so they
 * overlap the attention of chunk c.  The chunk launches follow each other
 * as in h3kv_attend (each may start on the SMs the previous one's tail
 * frees): a launch waits inside the kernel, bounded by the wait limit, for
 * a ready word in the scratch that the copy stream sets once the chunk's Q
 * rows are in and its O buffer is free.  The 4-byte values come from a 4 KB
 * pinned host table that the library allocates on the first call and keeps
 * until the process exits.  The result is bit-identical to h3kv_attend with
 * device Q and O and the same q_chunk and kv_block.
 *   Q_host: bf16 [store->heads, q_seq, 128]; O_host: fp32, same shape.
 *   scratch: device memory >= h3kv_hostio_scratch_bytes(store->heads,
 *   q_chunk), 16-byte aligned, caller-owned, reused by each call (calls that
 *   overlap on the GPU must not share it).
 * All work, copies included, is ordered after earlier work on `stream`, and
 * later work on `stream` sees O_host written.  Other arguments and errors as
 * h3kv_attend. */
h3kv_status h3kv_attend_hostio(const uint16_t *Q_host, int64_t q_seq, const h3kv_store *store, int32_t q_chunk,
                               int32_t kv_block, float softmax_scale, float *O_host, void *scratch,
                               size_t scratch_bytes, void *stream);

/* Size of the fixed device scratch that h3kv_attend_staged_static uses. */
#define H3KV_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* h3kv_attend_staged with no caller-provided scratch (no counterpart on the
 * kvi8r pages; it exists for callers that cannot allocate device memory -- a
 * plugin whose host application owns the whole device-memory budget, or code
 * on a path where a cudaMalloc, which can synchronise the device, is not
 * allowed).  The staging block and the per-row state live in a fixed
 * H3KV_STATIC_SCRATCH_BYTES array that the library holds on every GPU that
 * loads it, until the process exits.  The caller still passes Q, the store
 * and O; the library allocates nothing.
 *   Limit: round_up(h3kv_staging_bytes(store->heads, kv_block), 256)
 *          + store->heads * q_seq * 8  <=  H3KV_STATIC_SCRATCH_BYTES,
 *   otherwise H3KV_ERR_INVALID_ARG is returned before any device work.
 *   The first call on a device looks up the array's device address (with
 *   that device current); make that first call before any stream capture.
 *   Every call shares the array and leaves its contents behind; nothing in
 *   it needs to start at zero.  Calls that overlap on the GPU (other streams,
 *   other threads) race on it: run them one after another.
 * Results equal h3kv_attend_staged's. */
h3kv_status h3kv_attend_staged_static(const uint16_t *Q, int64_t q_seq, const h3kv_store *store,
                                      int32_t q_chunk, int32_t kv_block, float softmax_scale, float *O,
                                      void *stream);

/* ------------------------------------------------------------------ kvf8s
 * The kvf8s store: the kvi8s layout ("The K/V store options" table of the
 * Low VRAM write-up, kvi8s row; kv_store row of the H3 Streamed Blocks Inputs
 * table: K with one scale per 64-token block after mean smoothing, V fp8 per
 * channel, Q and K Hadamard-rotated, attended on the tensor cores straight
 * from the store) with fp8 e4m3 K in place of int8, so that both attention
 * products run on the fp8 tensor path.  e4m3 is the OCP E4M3 format (bias 7,
 * largest finite 448); every encode rounds to nearest even and saturates.
 *   K: k' = k H (the kvi8r basis); mu = the mean of k' over all seq tokens
 *      (per head and channel); per (head, 64-token block)
 *      s_k = max |k' - mu| / 448 over the block; codes e4m3((k' - mu) / s_k),
 *      all 0 where s_k == 0.  Subtracting mu shifts every score of a query
 *      row by the same amount, so attention does not need it; it is stored
 *      for inspection.
 *   V: not rotated; per (head, channel) s_v = max over all tokens |v| / 448;
 *      codes e4m3(v / s_v), the exact quotient rounded once (bit-exact
 *      for every channel whose absmax is at least 2^-100; below that the
 *      fp32 arithmetic can miss by one step), stored channel-major
 *      (V transposed) with a row stride of
 *      h3kv_f8_v_stride(seq) bytes; bytes of a row past seq are 0.
 *   The K (and query) codes are the same rounding of quotients of values
 *   that the kernels compute in fp32, formed as x * fp32(1/s).
 * Every buffer is caller-owned device memory, 16-byte aligned. */
typedef struct {
  uint8_t *k_codes;   /* e4m3 [heads, seq, 128] */
  uint8_t *v_codes_t; /* e4m3 [heads, 128, h3kv_f8_v_stride(seq)] */
  float *k_scales;    /* [heads, ceil(seq / H3KV_F8_K_BLOCK)] */
  float *v_scales;    /* [heads, 128] */
  float *k_mean;      /* [heads, 128] */
  int32_t heads;
  int64_t seq;
  int32_t head_dim;   /* must be 128 */
} h3kv_store_f8;

/* Tokens per K scale block of the kvf8s store. */
#define H3KV_F8_K_BLOCK 64

/* Row stride in bytes of the channel-major V codes: seq rounded up to a
 * multiple of 16 (0 for seq < 0). */
int64_t h3kv_f8_v_stride(int64_t seq);

/* Bytes of a kvf8s store's five buffers together (0 for invalid arguments). */
size_t h3kv_store_f8_bytes(int32_t heads, int64_t seq, int32_t head_dim);

/* Build the kvf8s store of bf16 K and V [heads, seq, 128] into `out`, whose
 * heads/seq/head_dim must match.  Two stream-ordered passes (statistics of
 * every head, then the encode); every reduction runs in a fixed order, so
 * the store is the same on every run.  heads <= 65535. */
h3kv_status h3kv_build_store_f8(const uint16_t *K, const uint16_t *V, int32_t heads, int64_t seq,
                                int32_t head_dim, const h3kv_store_f8 *out, void *stream);

/* kvf8s attention: q' = Q H; one fp32 scale per query row s_q = max|q'|/448
 * and e4m3 codes of q'/s_q; S = (Q codes . K codes) s_q s_k softmax_scale;
 * P = softmax(S) over all store->seq keys (non-causal), in kv_block-token
 * blocks combined by their log-sum-exp; O = P (V codes s_v).  V is not
 * rotated, so O needs no un-rotation.  Both products are e4m3 x e4m3 with
 * fp32 accumulation: the un-normalised softmax weights enter P.V as e4m3,
 * scaled so that the largest possible weight is 448.
 *   Q: bf16 [store->heads, q_seq, 128].  O: fp32 [store->heads, q_seq, 128].
 *   q_chunk, kv_block and softmax_scale as for h3kv_attend; the output is
 *   bit-identical for every q_chunk.  store->heads <= 65535. */
h3kv_status h3kv_attend_f8(const uint16_t *Q, int64_t q_seq, const h3kv_store_f8 *store, int32_t q_chunk,
                           int32_t kv_block, float softmax_scale, float *O, void *stream);

/* ------------------------------------------------------------------ kvfp4
 * The kvfp4 store: kvfp4s of the kv_store row of the H3 Streamed Blocks
 * Inputs table -- K/V kept as NVFP4 (e2m1 values with one e4m3 scale per 16
 * elements, 0.5625 byte per element), Q and K Hadamard-rotated, no K
 * smoothing and no query centring.  e2m1 has 1 sign, 2 exponent (bias 1) and
 * 1 mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.  e4m3 as for kvf8s.
 * For each (head, token) row x -- of K rotated (x = k H, the kvi8r basis) or
 * of V (not rotated) -- and each block B of 16 consecutive values:
 *   s_B = e4m3_rne(max_{j in B} |x_j| / 6)        (saturating at 448),
 *   c_j = e2m1_rne(x_j / s_B), sign of x_j        (saturating at +-6),
 *   every c_j = 0 where s_B == 0.
 * Codes are packed two per byte, element 2i in the low nibble of byte i.
 * Dequantisation c_j s_B is exact in fp16.  Every buffer is caller-owned
 * device memory, 16-byte aligned. */
typedef struct {
  uint8_t *k_codes;  /* e2m1 pairs [heads, seq, 64] */
  uint8_t *v_codes;  /* e2m1 pairs [heads, seq, 64] */
  uint8_t *k_scales; /* e4m3 [heads, seq, 8] */
  uint8_t *v_scales; /* e4m3 [heads, seq, 8] */
  int32_t heads;
  int64_t seq;
  int32_t head_dim;  /* must be 128 */
} h3kv_store_fp4;

/* Bytes of a kvfp4 store's four buffers together, 2 heads seq (64 + 8) (0
 * for invalid arguments). */
size_t h3kv_store_fp4_bytes(int32_t heads, int64_t seq, int32_t head_dim);

/* Build the kvfp4 store of bf16 K and V [heads, seq, 128] into `out`, whose
 * heads/seq/head_dim must match.  One stream-ordered pass; rows are
 * independent, so the store is the same on every run. */
h3kv_status h3kv_build_store_fp4(const uint16_t *K, const uint16_t *V, int32_t heads, int64_t seq,
                                 int32_t head_dim, const h3kv_store_fp4 *out, void *stream);

/* kvfp4 attention: q' = fp16(Q H); each K/V block of the store dequantised
 * to fp16 (exactly); S = q' K^T softmax_scale with fp32 accumulation;
 * P = softmax(S) over all store->seq keys (non-causal), in kv_block-token
 * blocks combined by their log-sum-exp, entering P.V as fp16; O = P V in
 * fp32.  V is not rotated, so O needs no un-rotation.
 *   Q: bf16 [store->heads, q_seq, 128].  O: fp32 [store->heads, q_seq, 128].
 *   q_chunk, kv_block and softmax_scale as for h3kv_attend; the output is
 *   bit-identical for every q_chunk. */
h3kv_status h3kv_attend_fp4(const uint16_t *Q, int64_t q_seq, const h3kv_store_fp4 *store, int32_t q_chunk,
                            int32_t kv_block, float softmax_scale, float *O, void *stream);

/* Synchronise `stream`, then return and clear the device error word that the
 * kernels set when a bounded wait runs out (H3KV_ERR_DEVICE_TIMEOUT), or
 * H3KV_ERR_CUDA if the synchronisation itself reports an error. */
h3kv_status h3kv_sync_status(void *stream);

/* Set the limit (nanoseconds) of every bounded in-kernel wait in later
 * launches; 0 restores the default of 1 s.  Process-wide.  A limit far below
 * the kernels' normal waits makes them give up early: the launch then
 * records H3KV_ERR_DEVICE_TIMEOUT, drains its own copies and MMAs, and exits
 * with its output undefined, leaving the context usable.  A wait whose
 * phase completes while its first (suspended) poll is pending never runs
 * out, however small the limit (see h3kv_debug_withhold_p). */
h3kv_status h3kv_set_wait_timeout_ns(uint64_t timeout_ns);

/* Diagnostic of the failure path (no counterpart on the pages): in later
 * attention launches (every path), the softmax warps of every CTA withhold
 * their "P ready" arrival for the 128-key tile `tile` of the launch (counted
 * from 0 within each launch), so that the MMA warp's bounded wait for it runs
 * out: the launch records H3KV_ERR_DEVICE_TIMEOUT, drains its copies and
 * MMAs and exits, its output undefined.  -1 (the default) withholds nothing;
 * below -1: H3KV_ERR_INVALID_ARG.  Process-wide.  A suspended barrier poll
 * can outlast a tiny wait limit, so a small limit alone does not make every
 * kernel give up; a wait on an arrival that never comes always runs out. */
h3kv_status h3kv_debug_withhold_p(int32_t tile);

/* Diagnostic of the failure path (no counterpart on the pages): launch one
 * CTA whose only wait is on a barrier that nothing ever arrives on, limited
 * to `timeout_ns` (0 = default).  The wait runs out, the kernel records
 * H3KV_ERR_DEVICE_TIMEOUT in the device error word and returns, so the next
 * h3kv_sync_status() on `stream` reports it.  Nothing faults or traps. */
h3kv_status h3kv_selftest_wait_timeout(uint64_t timeout_ns, void *stream);

/* Kernel launches that one h3kv_attend, h3kv_attend_exact, h3kv_attend_f8 or
 * h3kv_attend_fp4 call makes for `q_seq` query rows of `heads` heads over
 * `kv_seq` keys in chunks of `q_chunk` rows (0 for an empty call or a
 * non-positive argument).  With more than one head, at least 131072 keys and
 * at least 16 CTAs of 256 rows (more than 3840 rows) per head and chunk, the
 * call launches every chunk of head 0, then of head 1, and so on (heads x
 * chunks launches, each one head), so that the L2 keeps much of a head's
 * store between its chunks; otherwise one launch per chunk covers all heads.
 * Results do not depend on the order. */
int64_t h3kv_attend_launch_count(int64_t q_seq, int64_t kv_seq, int32_t heads, int32_t q_chunk);

/* Diagnostic of the reducing tensor-memory load (tcgen05.ld.red, sm_103a)
 * with which every attention path takes the row maximum of a full 128-key
 * tile: one CTA stores known fp32 values into 128 TMEM columns of each of its
 * 128 lanes, reloads them with the max reduction over each 32-column group,
 * and counts the reduced maxima that differ from the maxima of the stored
 * values plus the loaded values that differ from the stored ones.  Writes
 * the count to *mismatches (0 when the instruction behaves as the kernels
 * assume); synchronises `stream`.  NULL mismatches: H3KV_ERR_INVALID_ARG. */
h3kv_status h3kv_selftest_tmem_ld_max(int32_t *mismatches, void *stream);

/* Static description of a status code (never NULL). */
const char *h3kv_strerror(h3kv_status status);

#ifdef __cplusplus
}
#endif

#endif /* H3KV_H */
