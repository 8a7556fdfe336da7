/*
 * tq.h — C ABI of libtq: TurboQuant KV-cache quantisation over a paged cache,
 * written for NVIDIA GB300 (sm_103a).
 *
 * The method restated here comes from these pages:
 *   [vLLM-TQ]  "vLLM 源码完全拆解(十九):TurboQuant KV Cache 量化——Hadamard 旋转、
 *              Lloyd-Max 标量量化与分页缓存内核" (pinghaoyang.com.cn)
 *   [TQ-intro] "vLLM TurboQuant 介绍:极低比特 KV Cache 量化" (beaiera.top)
 *   [NVFP4-TQ] "NVIDIA KV Cache 量化中的 NVFP4 与 TurboQuant" (moonnryan.github.io)
 *
 * Two hot operations, and one for long cached histories:
 *   tq_store   per (token, KV head): L2 norm, normalised Walsh-Hadamard
 *              rotation, Lloyd-Max bucketize, norm-correction fold, bit-pack
 *              of the K indices (or an e4m3 cast for FP8 keys), asymmetric
 *              uniform quantisation of V, and one slot written into the paged
 *              cache through slot_mapping.
 *   tq_decode  attention for one query token per sequence read straight from
 *              the packed cache: split-K over partitions of the sequence with
 *              an online softmax, then an LSE-weighted reduce. No 16-bit copy
 *              of the cache is ever materialised.
 *   tq_dequant the cached keys and values expanded back to dense vectors in
 *              the original basis (continuation prefill over a long history).
 *
 * Conventions shared by every entry point
 *   - Ownership: the caller owns every buffer. The library allocates nothing,
 *     keeps no global state (except the fixed device array of
 *     tq_decode_noalloc below), never synchronises the stream and only
 *     enqueues kernels on the given stream (NULL = the legacy default stream).
 *   - Pointers documented "device" must be CUDA device memory of the current
 *     device; "host" pointers are plain CPU memory read during the call.
 *   - Errors detectable on the host return a negative tq_status before any
 *     launch. A launch failure returns TQ_ERR_CUDA. Data-dependent problems
 *     (a slot or block id out of range, a sequence longer than its block-table
 *     row) never trap: the offending item is skipped and a bit is OR-ed into
 *     the optional device status word (TQ_DEV_* below).
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t. */
typedef struct CUstream_st* tq_stream_t;

typedef enum {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = -1,        /* null pointer, bad size or count */
  TQ_ERR_UNSUPPORTED = -2,        /* shape or preset this build does not run */
  TQ_ERR_MISALIGNED = -3,         /* a pointer breaks its alignment rule */
  TQ_ERR_WORKSPACE_TOO_SMALL = -4,
  TQ_ERR_CUDA = -5                /* a kernel launch failed */
} tq_status;

/* Presets: [vLLM-TQ] section "TurboQuant 在 vLLM 中的位置", subsection
 * "四个预设对应什么" (TQ_PRESETS). */
typedef enum {
  TQ_PRESET_K8V4 = 0,     /* K: e4m3, no rotation, no norm; V: 4-bit        */
  TQ_PRESET_4BIT_NC = 1,  /* K: 4-bit Lloyd-Max + norm correction; V: 4-bit */
  TQ_PRESET_K3V4_NC = 2,  /* K: 3-bit Lloyd-Max + norm correction; V: 4-bit */
  TQ_PRESET_3BIT_NC = 3,  /* K: 3-bit + norm correction; V: 3-bit           */
  TQ_PRESET_PROD3 = 4     /* keys only: 2-bit Lloyd-Max code + 1-bit QJL residual
                             sign per coordinate (TurboQuant_prod; the tq_prod_*
                             entry points below, its own key cache)          */
} tq_preset;

typedef enum { TQ_DTYPE_F16 = 0, TQ_DTYPE_BF16 = 1, TQ_DTYPE_F32 = 2 } tq_dtype;

/* Bits OR-ed into *dev_status by the kernels. */
#define TQ_DEV_SLOT_OUT_OF_RANGE  1u  /* store: slot // block_size >= num_blocks   */
#define TQ_DEV_BLOCK_OUT_OF_RANGE 2u  /* decode: block id < 0 or >= num_blocks     */
#define TQ_DEV_SEQ_TOO_LONG       4u  /* decode: seq_len > max_seq_len or > row cap */
#define TQ_DEV_TIMEOUT            8u  /* decode: a bounded wait on a copy expired, or the
                                         launch's shared-memory plan did not fit */

/* Problem description shared by store and decode. */
typedef struct {
  int preset;            /* tq_preset                                        */
  int head_dim;          /* d; this build runs d = 128                        */
  int block_size;        /* tokens per cache block: 16, 32, 64 or 128         */
  int num_q_heads;       /* n_q (decode)                                      */
  int num_kv_heads;      /* n_kv; n_q % n_kv == 0 and n_q / n_kv <= 8         */
  int partition_tokens;  /* 0: a partial covers at most one whole sequence of
                            one KV head; > 0 (a multiple of 16): partials are
                            also cut every partition_tokens positions. Work is
                            split evenly over the GPU in either case.          */
  int flags;             /* OR of TQ_FLAG_* (0: none; unknown bits are an
                            error, TQ_ERR_INVALID_ARG)                         */
} tq_config;

/* tq_config.flags. TQ_FLAG_INDICES_READY: the caller guarantees that the
 * kernel launched immediately before tq_decode / tq_decode_partials on the
 * same stream writes neither seq_lens nor block_table (for example: they were
 * copied from the host earlier, and that kernel is tq_store or a projection).
 * The split kernel then reads them, and plans its work, before it waits for
 * that kernel (programmatic dependent launch), so the start-up chain lengths
 * -> block ids overlaps the previous kernel's tail. It still waits before it
 * reads q or the cache and before it writes anything. Breaking the guarantee
 * gives results computed from stale indices; no fault. */
#define TQ_FLAG_INDICES_READY 1

/* Byte layout of the paged cache (this library's ABI).
 *
 *   cache[num_blocks][n_kv][block_size / 16][tile_bytes]
 *
 * A tile holds 16 consecutive positions of one KV head, as separate regions:
 *   k_off     16 rows x k_row_bytes: the key's LSB-first index stream (bit
 *             b*i + j is bit j of index i; [vLLM-TQ] "位打包") or its e4m3 bytes
 *   v_off     16 x v_row_bytes: value index streams, taken in token pairs
 *             (2p, 2p+1) whose streams are interleaved in 16-bit words, four
 *             words per token in each 16-byte group: word i of token 2p+j is
 *             at v_off + 2p*v_row_bytes + 16*((i >> 2) ^ x) + 4*(i & 3) + 2j,
 *             x = 2*(p & 3) when v_row_bytes % 64 == 0 (a bank swizzle), else 0
 *   knorm_off 16 x fp16 stored key norms (-1 for FP8 keys)
 *   vscale_off, vzero_off   16 x fp16 value scales and zero points
 * so tile_bytes = 16 * slot_bytes and block_bytes = block_size * n_kv *
 * slot_bytes, the page size of [vLLM-TQ] "页内寻址:一页多少字节". Position p of
 * sequence b is in block block_table[b][p / block_size], row p % block_size.
 * Every region starts on a 16-byte boundary, so the kernels use 16-byte loads.
 */
typedef struct {
  int key_bits;           /* 3 or 4, or 8 for e4m3 keys                   */
  int value_bits;         /* 3 or 4                                        */
  int key_fp8;
  int norm_correction;
  int key_packed_bytes;   /* per token, pages' key_packed_size             */
  int value_packed_bytes; /* per token, pages' value_packed_size           */
  int slot_bytes;         /* key_packed_bytes + value_packed_bytes         */
  int tile_tokens;        /* 16                                            */
  int tile_bytes;
  int k_off, k_row_bytes;
  int v_off, v_row_bytes;
  int knorm_off, vscale_off, vzero_off;
  long long block_bytes;
} tq_layout;

/* Lloyd-Max codebook for N(0, 1/d): [vLLM-TQ] section "Lloyd-Max 量化器".
 * centroids ascending (num_levels = 2^bits of them), exactly antisymmetric,
 * fp32; midpoints[i] = fp32((c[i] + c[i+1]) / 2), the decision boundaries the
 * store compares against (a coordinate equal to a midpoint goes up). */
typedef struct {
  int head_dim;
  int bits;
  int num_levels;
  float centroids[16];
  float midpoints[15];
} tq_codebook;

/* Host. Solve the Lloyd-Max conditions for N(0, 1/head_dim) with `bits`
 * (1..4) levels: closed-form Gaussian conditional means iterated from the
 * uniform start on [-3.5 sigma, 3.5 sigma] to a 1e-13 change, symmetrised,
 * rounded to fp32. Deterministic. out: host, written on TQ_OK. */
tq_status tq_build_codebook(int head_dim, int bits, tq_codebook* out);

/* Host. Fill *out with the cache layout of cfg (see tq_layout). Returns
 * TQ_ERR_UNSUPPORTED for shapes the kernels do not run. */
tq_status tq_layout_for(const tq_config* cfg, tq_layout* out);

/* Device. Quantise and write num_tokens tokens into the cache.
 *   cfg, cb       host; cb must be tq_build_codebook(d, key_bits) (ignored
 *                 for TQ_PRESET_K8V4, may then be NULL)
 *   key, value    device, [num_tokens][n_kv][d] contiguous, in_dtype f16 or
 *                 bf16, 16-byte aligned
 *   slot_mapping  device int64 [num_tokens]; slot < 0 writes nothing
 *                 ([vLLM-TQ] "融合 kernel 的骨架"); slot s goes to block
 *                 s / block_size, row s % block_size
 *   cache         device, num_blocks * block_bytes bytes, 16-byte aligned
 *   dev_status    device uint32 or NULL
 * num_tokens == 0 is a no-op. Two tokens mapped to one slot race. */
tq_status tq_store(const tq_config* cfg, const tq_codebook* cb,
                   const void* key, const void* value, int in_dtype,
                   long long num_tokens, const long long* slot_mapping,
                   void* cache, long long num_blocks,
                   unsigned int* dev_status, tq_stream_t stream);

/* Host. Bytes of decode workspace for `batch` sequences of at most
 * max_seq_len tokens ([vLLM-TQ] "精度与性能", subsection "内存:workspace 预分配").
 * The decode splits the tile line of all (sequence, KV head) pairs evenly over
 * the warps of a persistent grid (at most 256 CTAs x 16 warps); each warp
 * writes one partial per segment it touches. A partial holds (acc / l) fp32
 * [d] and a log2-sum-exp fp32 for each of the n_q / n_kv query heads, and
 * there are at most batch * n_kv * P + 4096 of them, P = 1 when
 * partition_tokens is 0, else ceil(max_seq_len / partition_tokens).
 * Independent of the device. 0 on bad input. */
size_t tq_decode_workspace_size(const tq_config* cfg, int batch, int max_seq_len);

/* Device. out[b][h][:] = softmax_p(scale * q[b][h] . k_p) @ v_p over the
 * seq_lens[b] cached positions of sequence b, query head h reading KV head
 * h / (n_q / n_kv). Keys and values are read from the packed cache; the query
 * is rotated once ([vLLM-TQ] "读取内核", "分数计算:FP8 K 与 MSE K 的两条路径").
 *   q            device [batch][n_q][d], q_dtype f16 or bf16, 16-byte aligned
 *   cache        device, as written by tq_store
 *   block_table  device int32 [batch][bt_stride]
 *   seq_lens     device int32 [batch], each <= max_seq_len and
 *                <= bt_stride * block_size; 0 gives zeros
 *   scale        <= 0 selects 1/sqrt(d)
 *   out          device [batch][n_q][d] of out_dtype (f16, bf16 or f32),
 *                16-byte aligned
 *   workspace    device, >= tq_decode_workspace_size bytes, 16-byte aligned;
 *                its contents need no initialisation
 * Launches the split-K kernel then the reduce kernel on `stream`.
 * Like every kernel of this library they are launched with programmatic
 * dependent launch: each may be scheduled while the previous kernel in the
 * stream finishes, and waits for it (griddepcontrol.wait) before touching
 * any global memory, so stream order is kept for all arguments. */
tq_status tq_decode(const tq_config* cfg, const tq_codebook* cb,
                    const void* q, int q_dtype,
                    const void* cache, long long num_blocks,
                    const int* block_table, int bt_stride,
                    const int* seq_lens, int batch, int max_seq_len, float scale,
                    void* out, int out_dtype,
                    void* workspace, size_t workspace_bytes,
                    unsigned int* dev_status, tq_stream_t stream);

/* Device. One decode step with its new tokens: stores each sequence's newest
 * token into the cache, then returns what tq_decode returns over all
 * seq_lens[b] positions, the new one included. The pages run the step as a
 * cache write ([vLLM-TQ] "写入内核:store 路径如何旋转、量化与打包") followed by
 * the decode ([vLLM-TQ] "读取内核"); here both happen in the decode's split
 * kernel: the warp that reads the tile holding position seq_lens[b] - 1
 * quantises that token's key and value with the store's arithmetic, writes
 * them into the cache and uses them at once, so the step needs no separate
 * store launch.
 *   new_k, new_v  device [batch][n_kv][d], q_dtype, 16-byte aligned: the key
 *                 and value of position seq_lens[b] - 1 of sequence b
 *   cache         device, writable; row seq_lens[b] - 1 of each sequence ends
 *                 up holding exactly the bytes tq_store writes for that token
 *                 at slot block_table[b][p / block_size] * block_size +
 *                 p % block_size, p = seq_lens[b] - 1
 *   every other argument, layout and rule as for tq_decode (the workspace
 *   size is tq_decode_workspace_size's).
 * Not stored: sequences with seq_lens[b] == 0; sequences longer than
 * max_seq_len or bt_stride * block_size (TQ_DEV_SEQ_TOO_LONG, cut as in
 * tq_decode); a newest position whose block id is outside [0, num_blocks)
 * (TQ_DEV_BLOCK_OUT_OF_RANGE). Launches the split kernel then the reduce
 * kernel, like tq_decode. */
tq_status tq_decode_append(const tq_config* cfg, const tq_codebook* cb,
                           const void* q, int q_dtype,
                           const void* new_k, const void* new_v,
                           void* cache, long long num_blocks,
                           const int* block_table, int bt_stride,
                           const int* seq_lens, int batch, int max_seq_len, float scale,
                           void* out, int out_dtype,
                           void* workspace, size_t workspace_bytes,
                           unsigned int* dev_status, tq_stream_t stream);

/* The two stages of tq_decode, separately (same arguments and rules), for
 * callers that time or overlap them. tq_decode_partials writes only the
 * workspace; tq_decode_reduce reads it and writes out. */
tq_status tq_decode_partials(const tq_config* cfg, const tq_codebook* cb,
                             const void* q, int q_dtype,
                             const void* cache, long long num_blocks,
                             const int* block_table, int bt_stride,
                             const int* seq_lens, int batch, int max_seq_len,
                             float scale, void* workspace, size_t workspace_bytes,
                             unsigned int* dev_status, tq_stream_t stream);
tq_status tq_decode_reduce(const tq_config* cfg, const int* seq_lens, int batch,
                           int max_seq_len, int bt_stride, void* out, int out_dtype,
                           const void* workspace, size_t workspace_bytes,
                           tq_stream_t stream);

/* Device. tq_decode with no workspace argument: the same kernels, the same
 * result, with the workspace taken from a fixed array of
 * TQ_DECODE_NOALLOC_SCRATCH_BYTES that this library holds in device memory
 * (one copy per device). The method's description has no counterpart to this
 * call; it is an addition of this library for callers that cannot allocate
 * device memory: a plain C host with no device allocator of its own, or a
 * serving loop that must not call cudaMalloc between steps (cudaMalloc can
 * synchronise the device and can fail under memory pressure). Neither this
 * call nor the kernels it launches allocate host or device memory.
 *   Arguments, layouts and device-side errors are those of tq_decode.
 *   Limit: returns TQ_ERR_WORKSPACE_TOO_SMALL, launching nothing, when
 *   tq_decode_workspace_size(cfg, batch, max_seq_len) exceeds
 *   TQ_DECODE_NOALLOC_SCRATCH_BYTES (e.g. more than about 12,000 (sequence,
 *   KV head, partition) triples at 4 query heads per KV head).
 *   Set-up: every call looks the array's address up in the context current
 *   on the calling thread (a host-side look-up that allocates nothing). The
 *   first call in a context loads this part of the library there, which
 *   places the array in that device's memory; make that first call before
 *   any stream capture. Nothing is cached between calls, so a context that
 *   is reset or replaced simply gets its own array on its next first call.
 *   A failed look-up returns TQ_ERR_CUDA, launching nothing.
 *   Initial contents: nothing in the array needs to start at zero; each call
 *   writes every partial it later reads.
 *   Concurrency: all calls on one device share the one array, so two calls
 *   whose kernels may overlap (different streams, or different host threads
 *   without ordering between their streams) race and give wrong results.
 *   Calls on one stream run in order and are safe. */
#define TQ_DECODE_NOALLOC_SCRATCH_BYTES (32u << 20)
tq_status tq_decode_noalloc(const tq_config* cfg, const tq_codebook* cb,
                            const void* q, int q_dtype,
                            const void* cache, long long num_blocks,
                            const int* block_table, int bt_stride,
                            const int* seq_lens, int batch, int max_seq_len, float scale,
                            void* out, int out_dtype,
                            unsigned int* dev_status, tq_stream_t stream);

/* Device. The cached keys and values of `batch` sequences expanded back to
 * dense vectors in the original (unrotated) basis, for callers that run
 * attention outside this library over a long cached history (the pages'
 * continuation-prefill path: [vLLM-TQ] section "续写 prefill:小 chunk 走 decode,
 * 大 chunk 走反量化", subsection "反量化 kernel:_tq_full_dequant_kv"):
 *   index-coded keys  k = stored_norm * (H / sqrt(d)) c[idx]  (the rotation is
 *                     its own inverse)
 *   FP8 keys          k = e4m3 value
 *   values            v = fp16(scale) * code + fp16(zero)
 * computed in fp32 and rounded once to out_dtype.
 *   cfg, cb       host; as for tq_decode (cb ignored for TQ_PRESET_K8V4;
 *                 num_q_heads is not used)
 *   cache, num_blocks, block_table, bt_stride, seq_lens, batch, max_seq_len
 *                 device / sizes, exactly as for tq_decode
 *   key_out, value_out  device [batch][max_seq_len][n_kv][d] of out_dtype
 *                 (f16, bf16 or f32), 16-byte aligned, owned by the caller;
 *                 every element is written: positions at or past
 *                 min(seq_lens[b], max_seq_len, bt_stride * block_size) are 0
 *   dev_status    device uint32 or NULL: TQ_DEV_SEQ_TOO_LONG for a length
 *                 above that cap (the sequence is cut there),
 *                 TQ_DEV_BLOCK_OUT_OF_RANGE for a block id outside
 *                 [0, num_blocks) (its positions are written as 0)
 * batch == 0 or max_seq_len == 0 is a no-op. One launch: a CTA per
 * (sequence, 16-position tile, KV head), a half-warp per position; no
 * workspace. */
tq_status tq_dequant(const tq_config* cfg, const tq_codebook* cb,
                     const void* cache, long long num_blocks,
                     const int* block_table, int bt_stride,
                     const int* seq_lens, int batch, int max_seq_len,
                     void* key_out, void* value_out, int out_dtype,
                     unsigned int* dev_status, tq_stream_t stream);

/* ---- continuation chunks ---------------------------------------------
 * A prefill chunk of new tokens whose keys and values are already stored
 * (tq_store) attends to its sequence's cached history and to itself,
 * causally: [vLLM-TQ] section "续写 prefill:小 chunk 走 decode,大 chunk 走反量化"
 * (a chunk of at most 128 tokens is served by the decode kernel, query i as a
 * request of length cached + i + 1 over the sequence's block-table row). The
 * result equals tq_decode run once per query with those lengths; here one CTA
 * serves 64 / G queries of a KV head per pass over the history (G = n_q /
 * n_kv, which must divide 8), so the history is read ceil(q_len * G / 64)
 * times instead of q_len times.
 *
 * Host. Workspace bytes for `total_q` query rows whose sequences are at most
 * max_seq_len long: one record (d fp32 + an LSE) per (query, query head,
 * partition of partition_tokens positions, default 512). 0 for an invalid
 * config. */
size_t tq_continue_workspace_size(const tq_config* cfg, int total_q, int max_seq_len);

/* Device.
 *   cfg, cb       host; as for tq_decode (G = n_q / n_kv in {1, 2, 4, 8};
 *                 partition_tokens a multiple of 16 up to 4096, 0 = 512)
 *   q, q_dtype    device [total_q][n_q][d] f16 or bf16, 16-byte aligned: the
 *                 chunks' queries, sequence b's in rows
 *                 query_start[b] .. query_start[b + 1] - 1
 *   query_start   device int32 [batch + 1], non-decreasing, query_start[0] = 0
 *                 and query_start[batch] = total_q
 *   max_q_len     host; the longest chunk (rows of a longer chunk past
 *                 max_q_len are not served: they come out 0 and flag
 *                 TQ_DEV_SEQ_TOO_LONG)
 *   cache, num_blocks, block_table, bt_stride
 *                 as for tq_decode; row b of block_table is sequence b's
 *   seq_lens      device int32 [batch]: each sequence's length with its chunk
 *                 (query i of a chunk of q_len sits at position
 *                 seq_lens[b] - q_len + i and sees positions 0 .. that one)
 *   max_seq_len   host; >= every seq_lens[b] (sizes the partitions)
 *   scale         softmax scale; <= 0 means 1 / sqrt(d)
 *   out, out_dtype  device [total_q][n_q][d] f16, bf16 or f32, 16-byte
 *                 aligned, owned by the caller; every row is written (a
 *                 query that sees no position gives 0)
 *   workspace     device, >= tq_continue_workspace_size(cfg, total_q,
 *                 max_seq_len) bytes, 16-byte aligned, owned by the caller
 *   dev_status    device uint32 or NULL: TQ_DEV_SEQ_TOO_LONG for a length
 *                 above bt_stride * block_size or a chunk past max_q_len or
 *                 total_q, TQ_DEV_BLOCK_OUT_OF_RANGE for a bad block id (its
 *                 positions are skipped)
 * batch == 0, total_q == 0 or max_q_len == 0 is a no-op. Two launches: the
 * attention kernel (grid n_kv * ceil(max_q_len * G / 64) x partitions x
 * batch) and a reduce over the partitions. */
tq_status tq_continue(const tq_config* cfg, const tq_codebook* cb,
                      const void* q, int q_dtype,
                      const int* query_start, int batch, int total_q, int max_q_len,
                      const void* cache, long long num_blocks,
                      const int* block_table, int bt_stride,
                      const int* seq_lens, int max_seq_len, float scale,
                      void* out, int out_dtype,
                      void* workspace, size_t workspace_bytes,
                      unsigned int* dev_status, tq_stream_t stream);

/* ---- TurboQuant_prod keys (QJL residual) -------------------------------
 * The product-quantizer variant of the method: [vLLM-TQ] section "Lloyd-Max
 * 量化器" (the TurboQuant_mse / TurboQuant_prod passage; vLLM itself ships only
 * the MSE quantizer, section "TurboQuant 在 vLLM 中的位置", "为什么不用 QJL") and
 * [TQ-proj] the page on the open-source turboquant project
 * (kwkr.cn/news/555717), subsection "最后 1 bit 的巧思". For preset
 * TQ_PRESET_PROD3 a key k of n_kv heads is stored as
 *   n = ||k|| (fp16); y = (H / sqrt(d)) k / (n + 1e-8);
 *   idx = 2-bit Lloyd-Max code of y (codebook tq_build_codebook(d, 2));
 *   r = y - c[idx]; ||r|| (fp16); one bit per row i of S: (S r)_i >= 0
 * and <q, k> is estimated, without bias over a Gaussian S, as
 *   n * (<q_r, c[idx]> + ||r|| * sqrt(pi / 2) / d * <S q_r, signs>),
 * q_r = (H / sqrt(d)) q, signs in {-1, +1}. S is an input: d x d fp32,
 * row-major (row i is projection i), i.i.d. N(0, 1) entries drawn by the
 * caller; the same S must serve the store and the scores.
 *
 * Key cache (keys only): cache[num_blocks][n_kv][block_size / 16][tile_bytes],
 * a tile holding 16 positions of one KV head as regions: index streams
 * (16 x k_row_bytes, LSB-first), sign streams (16 x sign_row_bytes, bit i of
 * byte i / 8 is projection i), fp16 norms (16), fp16 residual norms (16). */
typedef struct {
  int mse_bits;           /* 2 */
  int slot_bytes;         /* per (position, KV head): 52 at d = 128 */
  int tile_bytes;         /* 16 * slot_bytes */
  int k_off, k_row_bytes;
  int sign_off, sign_row_bytes;
  int norm_off, rnorm_off;
  long long block_bytes;
} tq_prod_layout;

/* Host. The prod key cache layout of cfg (cfg->preset must be
 * TQ_PRESET_PROD3; num_q_heads is not used). */
tq_status tq_prod_layout_for(const tq_config* cfg, tq_prod_layout* out);

/* Device. Quantise and write num_tokens keys into the prod key cache.
 *   cb            host, tq_build_codebook(d, 2)
 *   S             device fp32 [d][d], row-major, 16-byte aligned
 *   key           device [num_tokens][n_kv][d], in_dtype f16 or bf16, 16-byte aligned
 *   slot_mapping  device int64 [num_tokens]; slot < 0 writes nothing
 *   cache         device, num_blocks * block_bytes, 16-byte aligned
 *   dev_status    device uint32 or NULL (TQ_DEV_SLOT_OUT_OF_RANGE)
 * Uses 129 KB of shared memory per CTA (S and a block of residuals). */
tq_status tq_prod_store(const tq_config* cfg, const tq_codebook* cb, const float* S,
                        const void* key, int in_dtype, long long num_tokens,
                        const long long* slot_mapping, void* cache, long long num_blocks,
                        unsigned int* dev_status, tq_stream_t stream);

/* Host. Workspace bytes of tq_prod_scores: the rotated query and S times it,
 * fp32, per (sequence, query head). 0 on bad input. */
size_t tq_prod_scores_workspace_size(const tq_config* cfg, int batch);

/* Device. scores[b][h][p] = scale * the estimate of <q[b][h], k_p> for every
 * cached position p < min(seq_lens[b], max_seq_len, bt_stride * block_size)
 * of sequence b, query head h reading KV head h / (n_q / n_kv); positions
 * from there to max_seq_len are written as 0.
 *   q            device [batch][n_q][d], q_dtype f16 or bf16, 16-byte aligned
 *   cache, num_blocks, block_table, bt_stride, seq_lens, batch, max_seq_len
 *                as for tq_decode (the prod key cache)
 *   scale        <= 0 selects 1 / sqrt(d)
 *   scores       device fp32 [batch][n_q][max_seq_len], 16-byte aligned
 *   workspace    device, >= tq_prod_scores_workspace_size bytes, 16-byte aligned
 *   dev_status   device uint32 or NULL (TQ_DEV_BLOCK_OUT_OF_RANGE,
 *                TQ_DEV_SEQ_TOO_LONG; a bad block's positions score 0)
 * Two launches: the query preparation, then the scores. */
tq_status tq_prod_scores(const tq_config* cfg, const tq_codebook* cb, const float* S,
                         const void* q, int q_dtype, const void* cache, long long num_blocks,
                         const int* block_table, int bt_stride, const int* seq_lens, int batch,
                         int max_seq_len, float scale, float* scores,
                         void* workspace, size_t workspace_bytes,
                         unsigned int* dev_status, tq_stream_t stream);

/* Host. Static description of a status code. */
const char* tq_status_string(int status);

/* Host. ABI version of this header (major * 100 + minor). */
int tq_version(void);

#define TQ_ABI_VERSION 105   /* 1.01: tq_dequant; 1.02: 3bit_nc runs; 1.03: TurboQuant_prod (tq_prod_*);
                                 1.04: tq_continue; 1.05: tq_decode_append */

#ifdef __cplusplus
}
#endif

#endif /* TQ_H_ */
