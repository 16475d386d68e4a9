/*
 * pa_decode.h -- C ABI of a GB300 (sm_103a) paged decode attention library
 * ("PagedAttention V2": partitioned online softmax followed by a
 * cross-partition log-sum-exp combine): single-query decode (pa_decode_v2,
 * pa_decode_v2_ex, pa_decode_v2_lse), multi-query decode (pa_decode_v2_mq),
 * E4M3 (fp8) caches (pa_decode_v2_fp8), host-resident per-step inputs
 * (pa_decode_v2_host_io) and a no-allocation variant
 * (pa_decode_v2_static_scratch).
 *
 * What it computes, per sequence s and query head h (the page
 * "paged_attention_v2_triton.py -- Triton PagedAttention V2 for BI-V100",
 * kernels `_paged_attn_v2_partition_kernel` and `_paged_attn_v2_reduce_kernel`
 * and the module docstring's Phase 2 formula):
 *
 *   kv   = h / (num_heads / num_kv_heads)                 (consecutive GQA groups)
 *   for t < L = seq_lens[s]:  b = block_tables[s, t / block_size], o = t % block_size
 *       K_t[d] = key_cache  [b, kv, d / x, o, d % x]      x = 16 / sizeof(element):
 *                                                         8 (fp16/bf16), 4 (fp32), 16 (E4M3)
 *       V_t[d] = value_cache[b, kv, d, o]
 *       z_t    = scale * sum_d query[s, h, d] * K_t[d]    (fp32)
 *   out[s, h, :] = sum_t softmax(z)_t * V_t               rounded to the element type
 *
 * computed in partitions of `partition_size` tokens: partition p holds tokens
 * [p*P, min((p+1)*P, L)) and yields (m_p, l_p, o_p) = (max z, sum e^(z - m_p),
 * normalised weighted V) -- phase 1, one persistent kernel; the partitions
 * are then combined with M = max m_p, w_p = e^(m_p - M) l_p / sum_q e^(m_q - M)
 * l_q, out = sum w_p o_p -- phase 2, a second kernel launched as a
 * programmatic dependent of the first (it starts while the first finishes and
 * waits for its results).  A sequence that fits in one partition is written
 * directly by phase 1 (single pass); a call in which no sequence can have two
 * partitions launches phase 1 only.
 * L = 0 yields zeros (the "flash_attention.metal" page's forward kernel takes
 * 1/l as 0 when l = 0).
 *
 * Memory: every pointer argument of pa_decode_v2 is a DEVICE pointer on the
 * current CUDA device; tensors are contiguous row-major.  The caller owns all
 * buffers.  The library reads query, caches, tables and lengths, and writes
 * `out` and `workspace` only.  Calls are enqueued on `stream` (a cudaStream_t,
 * NULL = legacy default stream) and never synchronise; results are ready when
 * the stream reaches that point.  Concurrent calls must not share a workspace.
 *
 * Errors: argument problems are reported by the return value before anything
 * is enqueued.  Problems only visible on the device (a block id outside
 * [0, num_blocks), seq_lens[s] outside [0, max_blocks_per_seq*block_size], a
 * bounded wait that ran out) are recorded in the workspace's error word, read
 * with pa_decode_v2_device_status(); the kernel never traps and never reads
 * outside the caches when it records a bad block id.
 */
#ifndef PA_DECODE_H
#define PA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types of query, caches and output. */
enum { PA_DTYPE_FP16 = 0, PA_DTYPE_BF16 = 1, PA_DTYPE_FP32 = 2 };

/* Status codes. */
enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, negative size, H % KH != 0, ... */
    PA_ERR_UNSUPPORTED = 2,   /* head_size not 64/80/96/112/128/256, block_size not
                                 8/16/32/64, partition_size not a positive multiple of
                                 block_size; a shape outside the chosen family (see
                                 pa_decode_v2_ex and pa_decode_v2_fp8) */
    PA_ERR_WORKSPACE = 3,     /* workspace smaller than pa_decode_v2_workspace_bytes() */
    PA_ERR_CUDA = 4,          /* a CUDA runtime call failed (launch, memset, ...) */
    PA_ERR_DEVICE_BOUNDS = 5, /* device-side: bad block id or sequence length */
    PA_ERR_TIMEOUT = 6        /* device-side: a bounded wait gave up */
};

/* Kernel families (pa_decode_v2_ex's `variant`). */
enum {
    PA_VARIANT_AUTO = 0,      /* SIMT when each kv head serves one query head (MHA), MMA otherwise */
    PA_VARIANT_SIMT = 1,      /* CUDA-core dot products and warp-shuffle reductions */
    PA_VARIANT_MMA = 2        /* mma.sync m16n8k16 over the [group x D] . [D x tokens] contraction */
};

/*
 * Bytes of device workspace pa_decode_v2 needs for these sizes: a 256-byte
 * header (error word, work counter, where a bounded wait gave up) and the
 * phase-1 partition states of the page's launcher -- max_logits
 * [S, H, Pmax] f32, exp_sums [S, H, Pmax] f32 and tmp_output
 * [S, H, Pmax, head_size] f32, with
 * Pmax = ceil(max_blocks_per_seq * block_size / partition_size).
 * Returns 0 for invalid sizes.
 */
size_t pa_decode_v2_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                    int max_blocks_per_seq, int block_size, int partition_size);

/*
 * Byte offsets of the workspace regions (for inspection in tests):
 * offsets[0] = max_logits (m_p, natural-log units, -inf for unused partitions),
 * offsets[1] = exp_sums (l_p, 0 for unused partitions),
 * offsets[2] = tmp_output (o_p, normalised; written only for sequences with
 *              more than one partition), offsets[3] = header (int32 error word
 *              at index 0), offsets[4] = total bytes.  *max_partitions = Pmax.
 * Returns PA_OK or PA_ERR_INVALID_ARG.
 */
int pa_decode_v2_workspace_layout(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                  int max_blocks_per_seq, int block_size, int partition_size,
                                  size_t offsets[5], int* max_partitions);

/*
 * Paged decode attention (see the top of this file).
 *   out          [num_seqs, num_heads, head_size]                      dtype, written
 *   query        [num_seqs, num_heads, head_size]                      dtype
 *   key_cache    [num_blocks, num_kv_heads, head_size/x, block_size, x] dtype,
 *                x = 16 / sizeof(element): 8 for fp16/bf16, 4 for fp32
 *   value_cache  [num_blocks, num_kv_heads, head_size, block_size]      dtype
 *   block_tables [num_seqs, max_blocks_per_seq] int32; entries past
 *                ceil(seq_lens[s]/block_size) are never read
 *   seq_lens     [num_seqs] int32, each in [0, max_blocks_per_seq*block_size]
 *   scale        softmax scale applied to q.k (fp32)
 *   dtype        PA_DTYPE_FP16, PA_DTYPE_BF16 or PA_DTYPE_FP32 (fp32 runs on the
 *                CUDA-core family, one query head per pass, every head size
 *                and block size, single- and multi-query; PA_ERR_UNSUPPORTED
 *                for the tensor-core variant and fp8 caches)
 *   stream       cudaStream_t to enqueue on
 *   max_blocks_per_seq  row stride of block_tables (the page's launcher reads
 *                it from the tensor's shape; a C ABI has to be told)
 *   num_blocks   number of physical blocks in each cache (bounds checks)
 *   workspace    device buffer of >= pa_decode_v2_workspace_bytes() bytes,
 *                16-byte aligned; NULL makes the call allocate and free one
 *                stream-ordered (cudaMallocAsync / cudaFreeAsync).  Its
 *                contents on entry do not matter: the call writes every byte
 *                of it that it reads.
 * out, query and the caches must be 16-byte aligned; tables 4-byte aligned.
 * With a workspace given, a call only enqueues kernels on `stream` (no
 * allocation, no synchronisation), so it can be captured into a CUDA graph
 * and replayed with new contents in its buffers (lengths up to the table's
 * capacity); the first call for a given shape should come before the capture.
 */
int pa_decode_v2(void* out, const void* query, const void* key_cache, const void* value_cache,
                 const int32_t* block_tables, const int32_t* seq_lens, float scale,
                 int num_seqs, int num_heads, int num_kv_heads, int head_size,
                 int block_size, int partition_size, int dtype, void* stream,
                 int max_blocks_per_seq, int num_blocks, void* workspace, size_t workspace_bytes);

/*
 * pa_decode_v2 with tuning controls, for tests and measurement.
 *   variant     PA_VARIANT_*; SIMT takes one query head per pass over the
 *               kv head's blocks (a group of G query heads takes G passes),
 *               MMA up to 8 query heads per pass (with G = 4, those of two kv
 *               heads, one block of each per pass; head sizes up to 128,
 *               blocks of 8, 16 or 32 tokens, an even kv-head count).  SIMT handles head sizes
 *               64/128/256 with blocks of 16 or 32 tokens, 80/96/112 with
 *               blocks of 16, 32 or 64, and 64/128 with blocks of 64, and
 *               fp32 in 8-token blocks at every head size (16-bit types in
 *               8-token blocks: PA_ERR_UNSUPPORTED); MMA every supported
 *               shape of the 16-bit types.  AUTO picks SIMT for G = 1 or fp32 where it
 *               applies, MMA otherwise.
 *   max_ctas    upper bound on the persistent grid (0 = one CTA per SM).
 *   timeout_ns  bound on every device-side wait (0 = 2^31 ns).
 * Results do not depend on variant-independent choices: for a fixed variant
 * the output is bitwise identical for every max_ctas.
 */
int pa_decode_v2_ex(void* out, const void* query, const void* key_cache, const void* value_cache,
                    const int32_t* block_tables, const int32_t* seq_lens, float scale,
                    int num_seqs, int num_heads, int num_kv_heads, int head_size,
                    int block_size, int partition_size, int dtype, void* stream,
                    int max_blocks_per_seq, int num_blocks, void* workspace, size_t workspace_bytes,
                    int variant, int max_ctas, long long timeout_ns);

/*
 * pa_decode_v2 that also returns, per (sequence, head), the log-sum-exp of
 * the scaled scores:
 *     lse[s * num_heads + h] = log( sum_t exp(scale * q[s,h] . k_t) )
 * over the sequence's seq_lens[s] tokens, natural log, fp32; -INFINITY for a
 * sequence with no tokens.  It is the value the forward kernel of the page
 * "flash_attention.metal -- Flash Attention Metal Shaders" stores beside its
 * output (its running maximum plus the log of its running sum, "log-sum-exp
 * for backward pass"), reached here by the same cross-partition combine as
 * the output (page "paged_attention_v2_triton.py -- Triton PagedAttention V2
 * for BI-V100", module docstring: M = max m_p, total = sum exp(m_p - M) l_p,
 * lse = M + log total).  With it, outputs computed over disjoint token sets
 * (for example the two halves of a sequence split across calls or devices)
 * merge exactly: out = sum_i exp(lse_i - LSE) out_i, LSE = log sum_i exp(lse_i).
 *   lse   DEVICE buffer of num_seqs * num_heads floats, 4-byte aligned, written
 *         (NULL: behaves as pa_decode_v2).
 * Every other argument, the ownership and the errors are those of
 * pa_decode_v2 (the kernel family is chosen as PA_VARIANT_AUTO); a misaligned
 * lse is PA_ERR_INVALID_ARG.
 */
int pa_decode_v2_lse(void* out, float* lse, const void* query, const void* key_cache,
                     const void* value_cache, const int32_t* block_tables, const int32_t* seq_lens,
                     float scale, int num_seqs, int num_heads, int num_kv_heads, int head_size,
                     int block_size, int partition_size, int dtype, void* stream,
                     int max_blocks_per_seq, int num_blocks, void* workspace, size_t workspace_bytes);

/*
 * pa_decode_v2_lse over an fp8 KV cache.  The launcher of page
 * "paged_attention_v2_triton.py -- Triton PagedAttention V2 for BI-V100" takes
 * kv_cache_dtype, k_scale and v_scale (and ignores them); here the caches hold
 * E4M3 codes ("e4m3fn": sign, 4 exponent bits with bias 7, 3 fraction bits,
 * no infinities, code 0x7f/0xff NaN) and the real keys and values are
 * k_scale * K and v_scale * V.  With one-byte elements the key layout's x is
 * 16 (16 bytes per chunk, as the launcher's x_pack = key_cache.shape[-1]):
 *   key_cache    [num_blocks, num_kv_heads, head_size/16, block_size, 16] uint8
 *   value_cache  [num_blocks, num_kv_heads, head_size, block_size]        uint8
 *   query, out   [num_seqs, num_heads, head_size]   dtype (fp16 or bf16)
 *   k_scale, v_scale   finite fp32 multipliers (PA_ERR_INVALID_ARG otherwise)
 * Every other argument, the workspace, ownership and errors are those of
 * pa_decode_v2_lse.  The tensor-core kernel family runs every group size
 * and every shape pa_decode_v2 takes: head_size 64, 80, 96, 112, 128 or 256,
 * block_size 8, 16, 32 or 64 (PA_ERR_UNSUPPORTED otherwise).
 */
int pa_decode_v2_fp8(void* out, float* lse, const void* query, const void* key_cache,
                     const void* value_cache, const int32_t* block_tables, const int32_t* seq_lens,
                     float scale, float k_scale, float v_scale, int num_seqs, int num_heads,
                     int num_kv_heads, int head_size, int block_size, int partition_size, int dtype,
                     void* stream, int max_blocks_per_seq, int num_blocks, void* workspace,
                     size_t workspace_bytes);

/*
 * Multi-query decode: q_len new tokens per sequence (speculative or
 * multi-token-prediction verification), each query row attending causally.
 * The decode of page "paged_attention_v2_triton.py -- Triton PagedAttention V2
 * for BI-V100" is its one-row case (module docstring: "For decode
 * (BLOCK_M=1), the Q tile is just one vector"); q_len > 1 rows follow the
 * causal rule of the prefix-prefill kernel its paged gather comes from: the
 * sequence's last q_len cached tokens are the new ones, and query row i sits
 * at position L - q_len + i (L = seq_lens[s]) and attends to positions
 * 0 .. L - q_len + i.  Their K and V must already be in the cache.
 *   query, out  [num_seqs, q_len, num_heads, head_size]   dtype
 *   lse         NULL, or DEVICE [num_seqs, q_len, num_heads] fp32 (as in
 *               pa_decode_v2_lse), written
 *   seq_lens    [num_seqs] int32, each in [q_len, max_blocks_per_seq*block_size]
 *               (a length below q_len is recorded as PA_ERR_DEVICE_BOUNDS)
 *   q_len       1 .. 1024 (q_len = 1 is pa_decode_v2_lse)
 *   workspace   >= pa_decode_v2_workspace_bytes(num_seqs * q_len, ...) bytes, or NULL
 * The other arguments, ownership and errors are those of pa_decode_v2 (kernel
 * family chosen as PA_VARIANT_AUTO).  The q_len query rows of a sequence share
 * its K/V loads: each kv head's q_len * (num_heads / num_kv_heads) rows are
 * the rows of the tensor-core product (8 or 16 per work unit), each masked to
 * the positions it may see; fp32 rows run on the CUDA-core family, one row
 * per pass.
 */
int pa_decode_v2_mq(void* out, float* lse, const void* query, const void* key_cache,
                    const void* value_cache, const int32_t* block_tables, const int32_t* seq_lens,
                    float scale, int num_seqs, int q_len, int num_heads, int num_kv_heads,
                    int head_size, int block_size, int partition_size, int dtype, void* stream,
                    int max_blocks_per_seq, int num_blocks, void* workspace, size_t workspace_bytes);

/*
 * Multi-query decode over an fp8 (E4M3) KV cache: the q_len causal query rows
 * of pa_decode_v2_mq (row i of sequence s sits at position L - q_len + i and
 * sees positions 0 .. L - q_len + i) with the caches, scales and element
 * reading of pa_decode_v2_fp8 (the launcher of "paged_attention_v2_triton.py
 * -- Triton PagedAttention V2 for BI-V100" takes kv_cache_dtype, k_scale and
 * v_scale whatever the query rows).
 *   query, out   [num_seqs, q_len, num_heads, head_size]   dtype (fp16 or bf16)
 *   key_cache    [num_blocks, num_kv_heads, head_size/16, block_size, 16] uint8
 *   value_cache  [num_blocks, num_kv_heads, head_size, block_size]        uint8
 *   lse          NULL, or DEVICE [num_seqs, q_len, num_heads] fp32, written
 *   k_scale, v_scale   finite fp32 multipliers (PA_ERR_INVALID_ARG otherwise)
 *   seq_lens     each in [q_len, max_blocks_per_seq*block_size]
 *   workspace    >= pa_decode_v2_workspace_bytes(num_seqs * q_len, ...) bytes, or NULL
 * Shapes as for pa_decode_v2_fp8 (PA_ERR_UNSUPPORTED otherwise); every other
 * argument, the ownership and the errors are those of pa_decode_v2_mq.
 */
int pa_decode_v2_mq_fp8(void* out, float* lse, const void* query, const void* key_cache,
                        const void* value_cache, const int32_t* block_tables, const int32_t* seq_lens,
                        float scale, float k_scale, float v_scale, int num_seqs, int q_len,
                        int num_heads, int num_kv_heads, int head_size, int block_size,
                        int partition_size, int dtype, void* stream, int max_blocks_per_seq,
                        int num_blocks, void* workspace, size_t workspace_bytes);

/*
 * Bytes of device workspace pa_decode_v2_host_io needs: the workspace of
 * pa_decode_v2 plus device staging for query, out (room for 4-byte elements,
 * whatever the dtype), block_tables and seq_lens.  Returns 0 for invalid sizes.
 */
size_t pa_decode_v2_host_io_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads,
                                            int head_size, int max_blocks_per_seq, int block_size,
                                            int partition_size);

/*
 * pa_decode_v2 for callers that hold the per-step inputs in HOST memory (a
 * serving loop): query_host, block_tables_host and seq_lens_host are copied
 * into device staging inside `workspace`, the decode runs on the device-
 * resident caches (key_cache, value_cache: DEVICE pointers), and the result is
 * copied back into out_host.  Everything is enqueued on `stream` with
 * cudaMemcpyAsync; the call returns without synchronising, so the host buffers
 * must stay alive and untouched until the stream has passed this call (use
 * page-locked host memory for the copies to be asynchronous).  `workspace`
 * (DEVICE, 16-byte aligned, >= pa_decode_v2_host_io_workspace_bytes()) is
 * required.  Sizes, layouts and status codes as for pa_decode_v2.
 */
int pa_decode_v2_host_io(void* out_host, const void* query_host, const void* key_cache,
                         const void* value_cache, const int32_t* block_tables_host,
                         const int32_t* seq_lens_host, float scale, int num_seqs, int num_heads,
                         int num_kv_heads, int head_size, int block_size, int partition_size,
                         int dtype, void* stream, int max_blocks_per_seq, int num_blocks,
                         void* workspace, size_t workspace_bytes);

/*
 * Size of the scratch array behind pa_decode_v2_static_scratch: 32 MiB of
 * device memory, reserved on every device that loads the library, for as long
 * as the process lives.
 */
#define PA_DECODE_V2_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * pa_decode_v2 for callers that must not allocate device memory at call time.
 * The pages have no counterpart: this is a deployment aid of this library.
 *
 * Who needs it: a process whose device memory is all reserved in advance by
 * another allocator (so a new cudaMalloc would fail), a latency-critical loop
 * that cannot risk an allocation call synchronising the device or stalling
 * other streams, or a deployment that fixes its memory footprint at start-up
 * and forbids allocation afterwards.  Such callers can use neither a
 * workspace of their own nor the library's stream-ordered allocation.
 *
 * What it does: the same computation as pa_decode_v2 (same arguments, minus
 * the workspace), with the scratch taken from a fixed array of
 * PA_DECODE_V2_STATIC_SCRATCH_BYTES inside the library's device memory.  It
 * calls no cudaMalloc, cudaFree or other allocating routine.  The caller
 * still provides all inputs and `out`.
 *   - Sizes whose workspace (pa_decode_v2_workspace_bytes) exceeds the array
 *     are rejected with PA_ERR_WORKSPACE before anything is enqueued.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it with the
 *     id of the device's context; make that first call before any stream
 *     capture.  If the context is destroyed and recreated (cudaDeviceReset),
 *     the array is a new one: the next call sees the new context id and looks
 *     the address up again, so make that call before any capture too.  (The
 *     array's contents do not survive the reset; nothing relies on them.)
 *   - All calls on a device share the one array, which keeps the last call's
 *     contents; the counters that must start at zero are cleared by each call
 *     on its stream.  Calls whose execution overlaps on the GPU (different
 *     streams, or threads without ordering between them) race on the array
 *     and give undefined results: order them on one stream.
 * Status codes as for pa_decode_v2.
 */
int pa_decode_v2_static_scratch(void* out, const void* query, const void* key_cache,
                                const void* value_cache, const int32_t* block_tables,
                                const int32_t* seq_lens, float scale, int num_seqs, int num_heads,
                                int num_kv_heads, int head_size, int block_size, int partition_size,
                                int dtype, void* stream, int max_blocks_per_seq, int num_blocks);

/*
 * Device-side status of the last call that used `workspace`: synchronises
 * `stream`, copies the error word and stores it in *status (PA_OK if none).
 * Returns PA_OK, or PA_ERR_CUDA if the copy or the synchronisation failed.
 */
int pa_decode_v2_device_status(const void* workspace, void* stream, int* status);

/* Static description of a status code. */
const char* pa_decode_v2_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* PA_DECODE_H */
