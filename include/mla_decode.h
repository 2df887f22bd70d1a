/*
 * mla_decode.h -- C ABI of libmla_decode: absorbed ("forward_mqa") Multi-head
 * Latent Attention decode over a paged latent KV cache, for GB300 (sm_103a).
 *
 * What it computes. For request b with L = seq_lens[b] cached tokens and each
 * head h < N:
 *     K[t]   = latent_cache[block_table[b, t / page_size], t % page_size, 0:576]
 *     V[t]   = K[t][0:512]
 *     s[t]   = softmax_scale * dot(q[b, h, 0:576], K[t])
 *     lse    = ln sum_t exp(s[t])
 *     out    = sum_t exp(s[t] - lse) * V[t]
 * This is the data-movement friendly MLA path: MQA with QK head dim Lkv+R and
 * V head dim Lkv, sdpa(cat[ql_nope, q_pe], cat[kv_c, k_pe], kv_c)
 * (vLLM "mla_attention" API docs, module docstring, "Data-Movement Friendly
 * Approach (i.e. forward_mqa)"). The problem statement and argument list
 * follow ModelOpt "modelopt.torch.kernels.quantization.attention.mla",
 * mla_attention_decode (q, latent_cache, block_table, b_seq_len,
 * softmax_scale, kv_lora_rank, qk_rope_head_dim, page_size, num_kv_splits,
 * return_lse). The cache layout [num_blocks, block_size, head_size] with one
 * latent KV head is vLLM mla/common.py (vllm-cpu 0.8.5.post2),
 * MLACommonBackend.get_kv_cache_shape.
 *
 * Conventions for every entry point.
 *   - All device pointers are caller-owned; the library never allocates or
 *     frees device memory. Scratch space is the caller's `workspace`, sized
 *     by mla_decode_plan (mla_decode_noalloc instead uses a fixed array
 *     inside the library, see its comment).
 *   - Every call returns an int status: MLA_OK (0) or a negative MLA_ERR_*.
 *     Argument errors are detected on the host before anything is enqueued.
 *   - Device work is enqueued asynchronously on `stream` (a cudaStream_t
 *     passed as void*, NULL = legacy default stream). No entry point except
 *     mla_read_error synchronises the host with the device, so mla_decode can
 *     be captured in a CUDA graph.
 *   - Errors the device detects (a block id outside [0, num_blocks), a
 *     seq_len longer than the block table allows) are recorded in a status
 *     word at the start of `workspace`; the offending page is treated as
 *     absent. Nothing traps. Read them with mla_read_error.
 *   - Supported shapes: kv_lora_rank = 512, rope_dim = 64, page_size = 64,
 *     1 <= num_heads <= 128. Anything else returns MLA_ERR_UNSUPPORTED.
 *   - bf16 data are raw IEEE bfloat16 bit patterns (uint16), little endian.
 */
#ifndef MLA_DECODE_H
#define MLA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_DECODE_ABI_VERSION 5

/* Status codes. */
#define MLA_OK                 0
#define MLA_ERR_INVALID_ARG   -1  /* null pointer, negative size, inconsistent plan */
#define MLA_ERR_UNSUPPORTED   -2  /* shape outside the supported set */
#define MLA_ERR_WORKSPACE     -3  /* workspace missing, too small or misaligned */
#define MLA_ERR_CUDA          -4  /* a CUDA runtime call or launch failed */
#define MLA_ERR_BAD_BLOCK_ID  -5  /* device: block_table entry outside [0, num_blocks) */
#define MLA_ERR_BAD_SEQ_LEN   -6  /* device: seq_len < 0 or > max_blocks_per_seq*page_size */
#define MLA_ERR_TIMEOUT       -7  /* device: a bounded wait inside a kernel expired */
#define MLA_ERR_SCRATCH_LIMIT -8  /* mla_decode_noalloc: plan needs more than its fixed scratch */
#define MLA_ERR_RANGE         -9  /* device: mla_decode_fp8 saw a q entry beyond +-65504 */

/* Kernel variants the planner can choose (mla_decode_plan_t.kernel). */
#define MLA_KERNEL_SIMT   1  /* CUDA-core split kernel, any 1 <= N <= 128 */
#define MLA_KERNEL_TC     2  /* tcgen05/TMEM + TMA CTA-pair kernel, heads padded to 128 */

/* Plan flags (mla_decode_plan_t.flags, and the `flags` argument). */
#define MLA_PLAN_FORCE_SIMT  0x1u  /* use MLA_KERNEL_SIMT even where MLA_KERNEL_TC applies */
#define MLA_PLAN_SPLIT_ONLY  0x2u  /* never choose the page-balanced schedule */
#define MLA_PLAN_FORCE_BALANCED 0x4u  /* with num_kv_splits = 0: the page-balanced schedule
                                         wherever it applies, whatever the estimate */
#define MLA_PLAN_FP32_PARTIALS 0x8u  /* keep the split schedule's partial rows in fp32 (default
                                        bf16, the precision of the decode's output) */
/* Test only (failure detection without a fault): the tensor-core kernel's
 * CTA 0 never issues its first K-ring load and every bounded wait of the call
 * is shortened to 2 ms (the merge's to 8 ms). The score warp's wait for that
 * load runs out, the call records MLA_ERR_TIMEOUT with detail 8 (that wait
 * site), every role drains its own loads and MMAs, TMEM is freed and the
 * kernel returns; the context stays usable. Never set in normal use. */
#define MLA_PLAN_DEBUG_WITHHOLD_LOAD 0x100u

/*
 * A decode plan: the sizes, the schedule and the kernel variant. It is plain
 * data computed on the host; mla_decode reads it, never changes it, and
 * rejects (MLA_ERR_INVALID_ARG) a plan whose launch shape or workspace layout
 * does not follow from its sizes.
 *
 * Split schedule (sched_pairs == 0; ModelOpt mla_attention_decode,
 * num_kv_splits: a fixed split count along the token axis). Split s of
 * request b covers tokens [s*C_b, min((s+1)*C_b, L_b)) with
 * C_b = page_size * ceil(ceil(L_b/page_size)/S); empty splits contribute
 * nothing. With S = 1 the decode kernel writes `out` and `lse` itself; with
 * S > 1 it writes partial rows [B,N,S,Lkv] (each normalised by its own
 * weights; bf16, rounded to nearest even like the final output, or fp32 with
 * MLA_PLAN_FP32_PARTIALS) and their fp32 LSEs [B,N,S] into the workspace,
 * and the LSE-weighted merge combines them in fp32 (an empty split writes
 * only its LSE, -inf: its weight is 0 and its row is never read). The tensor-core kernel runs
 * min(B*S, num_sms/2) CTA pairs, each over a contiguous run of the B*S
 * (request, split) items in request-major order, and stages a request's q
 * once for the consecutive splits it takes.
 *
 * Page-balanced schedule (sched_pairs = C > 0, MLA_KERNEL_TC, B <= 512,
 * num_kv_splits = 1). This is a work-partitioning choice of this library; the
 * papers' split-KV has no counterpart of it. In work units, a request with
 * p > 0 pages is 5 units of fixed cost followed by its p pages (an empty
 * request is nothing); the batch's units, request after request (taken from
 * the device seq_lens at run time, T in total), are cut into C contiguous
 * ranges, range c = units [floor(c*T/C), floor((c+1)*T/C)), one per CTA
 * pair. A request whose pages lie inside one range is written directly; one
 * whose pages cross range boundaries leaves fp32 partial rows ([2C,N,Lkv] /
 * [2C,N] in the workspace: slot 2c for the first request with pages in range
 * c, slot 2c+1 for its last) that a second kernel combines with the
 * LSE-weighted merge. Results agree with the split schedule up to rounding.
 */
typedef struct mla_decode_plan {
    int32_t  batch;               /* B */
    int32_t  num_heads;           /* N */
    int32_t  kv_lora_rank;        /* Lkv = 512 */
    int32_t  rope_dim;            /* R = 64 */
    int32_t  page_size;           /* tokens per block = 64 */
    int32_t  max_blocks_per_seq;  /* block_table row length */
    int32_t  max_seq_len;         /* upper bound of seq_lens used for planning */
    int32_t  num_kv_splits;       /* S used by mla_decode, >= 1 */
    int32_t  kernel;              /* MLA_KERNEL_* */
    int32_t  num_sms;             /* SM count the plan was made for */
    int32_t  grid_ctas;           /* CTAs the decode kernel launches */
    uint32_t flags;               /* MLA_PLAN_* as requested */
    uint64_t workspace_bytes;     /* bytes of `workspace` mla_decode needs */
    uint64_t partial_offset;      /* byte offset of o_part [B,N,S,Lkv] (bf16, or fp32) */
    uint64_t lse_partial_offset;  /* byte offset of lse_part [B,N,S] fp32 */
    int32_t  sched_pairs;         /* 0: split schedule; C > 0: page-balanced schedule */
    uint32_t reserved[7];
} mla_decode_plan_t;

/*
 * mla_decode_plan -- choose S and the kernel, size the workspace. Host only.
 *
 *   batch, num_heads           B >= 0, 1 <= N <= 128.
 *   kv_lora_rank, rope_dim     must be 512 and 64.
 *   page_size                  must be 64.
 *   max_blocks_per_seq         block_table row length, >= 1.
 *   max_seq_len                upper bound of every seq_lens[b] (0..max_blocks_per_seq*page_size).
 *   seq_lens_host              optional host copy of seq_lens [B] (NULL allowed);
 *                              when given, the planner sizes S from the real lengths.
 *   num_kv_splits              S > 0 is used as given (fixed, batch-invariant);
 *                              0 lets the planner choose S, or the page-balanced
 *                              schedule over num_sms/2 CTA pairs (MLA_KERNEL_TC,
 *                              B <= 512, unless MLA_PLAN_SPLIT_ONLY), from its
 *                              cost estimate.
 *   num_sms                    SMs of the target device (152 on GB300), >= 1.
 *   flags                      MLA_PLAN_* bits.
 *   plan                       out: filled on MLA_OK.
 */
int mla_decode_plan(int batch, int num_heads, int kv_lora_rank, int rope_dim,
                    int page_size, int max_blocks_per_seq, int max_seq_len,
                    const int32_t* seq_lens_host, int num_kv_splits, int num_sms,
                    uint32_t flags, mla_decode_plan_t* plan);

/*
 * mla_workspace_init -- zero the status header of a fresh workspace
 * (cudaMemsetAsync of its first 8192 bytes on `stream`: the status word and
 * the per-request counters through which the page-balanced merge learns that
 * a request's partial rows are complete; every call leaves the counters at
 * zero). Call once per workspace allocation before its first mla_decode, and
 * again after a call that reported MLA_ERR_TIMEOUT (an abandoned call may
 * leave counters behind).
 */
int mla_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * mla_decode -- absorbed MLA decode (the `forward_mqa` of the vLLM pages).
 *
 *   plan             from mla_decode_plan with the same B, N, max_blocks_per_seq.
 *   q                device, bf16 [B, N, 576] contiguous: [ql_nope (512) | q_pe (64)]
 *                    (vLLM mla_attention API docs, MLAAttention.forward_impl:
 *                    mqa_q = cat(ql_nope, q_pe)). 16-byte aligned.
 *   latent_cache     device, bf16 [num_blocks, 64, 576] contiguous:
 *                    [kv_c (512) | k_pe (64)] per token. 16-byte aligned.
 *   num_blocks       blocks in latent_cache, >= 1.
 *   block_table      device, int32 [B, max_blocks_per_seq]; entries past
 *                    ceil(L_b/64) are never read.
 *   seq_lens         device, int32 [B]; rows past L_b in the last page are
 *                    never read or weighted.
 *   softmax_scale    multiplies q.K before the softmax (the model's
 *                    qk_head_dim**-0.5, times mscale^2 under yarn RoPE).
 *   out              device, bf16 [B, N, 512]; rounded to nearest even.
 *   lse              device, fp32 [B, N], natural log of sum exp(scaled
 *                    scores); NULL skips it (return_lse=False). An empty
 *                    request (L_b = 0) gives out = 0, lse = -inf.
 *   workspace        device, >= plan->workspace_bytes, 256-byte aligned,
 *                    initialised once with mla_workspace_init.
 *   stream           cudaStream_t as void*.
 * Calls that share a workspace must not overlap on the device.
 */
int mla_decode(const mla_decode_plan_t* plan, const void* q, const void* latent_cache,
               int64_t num_blocks, const int32_t* block_table, const int32_t* seq_lens,
               float softmax_scale, void* out, float* lse,
               void* workspace, size_t workspace_bytes, void* stream);

/*
 * mla_decode_fp8 -- mla_decode over an fp8 latent cache: E4M3 codes with one
 * per-tensor scale (vLLM mla_attention API docs, MLAAttention.forward_impl:
 * an fp8 cache other than fp8_ds_mla is viewed as the platform's fp8 dtype
 * and read with the layer's _k_scale; raon-1-mini MLA page,
 * _attn_read_kv_cache: a plain per-tensor fp8 cache is read as E4M3). Entry
 * t of the cache is k_scale * e4m3(code): K[t] all 576 of them, V[t] the
 * first 512. The query stays bf16 and the outputs are as for mla_decode.
 *
 *   plan            from mla_decode_plan (the same plans as mla_decode; it
 *                   must use MLA_KERNEL_TC, else MLA_ERR_UNSUPPORTED).
 *   latent_cache_fp8  device, uint8 [num_blocks, 64, 576] E4M3 codes
 *                   (OCP 8-bit floating point E4M3: sign, 4 exponent bits with
 *                   bias 7, 3 mantissa bits, no infinities, 0x7F/0xFF NaN),
 *                   16-byte aligned. 36,864 bytes per page.
 *   k_scale         finite, > 0.
 *   q               bf16 [B, N, 576]; every entry within +-65504 (the kernel
 *                   multiplies in f16, into which every E4M3 value and every
 *                   such bf16 value convert exactly; a larger entry is
 *                   recorded as MLA_ERR_RANGE, detail = its request).
 *   other arguments as for mla_decode.
 * The tensor cores take f16 operands (q, the widened cache entries and the
 * softmax weights, which are rounded to f16 instead of bf16); everything else
 * is the arithmetic of mla_decode.
 */
int mla_decode_fp8(const mla_decode_plan_t* plan, const void* q, const void* latent_cache_fp8,
                   int64_t num_blocks, const int32_t* block_table, const int32_t* seq_lens,
                   float softmax_scale, float k_scale, void* out, float* lse,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * mla_decode_noalloc -- mla_decode for callers that cannot allocate device
 * memory. The pages have no counterpart to this entry point.
 *
 * Who needs it: code that may not allocate while it runs (an allocation can
 * synchronise the device, and many serving loops forbid it), runtimes that
 * hand out all device memory from their own pools and have no allocator to
 * offer, and bindings that can pass only the operation's own tensors. Such a
 * caller passes the inputs and outputs of mla_decode and no workspace.
 *
 * Scratch: the status words, the page-balanced merge's counters and the
 * partial rows live in one fixed device array of 32 MiB inside the library;
 * every GPU that loads the library holds it until the process exits. A plan
 * whose workspace_bytes exceeds 32 MiB is rejected with MLA_ERR_SCRATCH_LIMIT.
 * 8 KiB go to the status header; a split-schedule row (request, head,
 * split) takes 1,028 bytes (2,052 with MLA_PLAN_FP32_PARTIALS) and a
 * page-balanced row 2,052: up to 32,632 split rows fit (B*N*S: e.g. B=32,
 * N=128, S=7 fits and S=8 does not; with fp32 rows 16,348: S=3 fits, S=4
 * does not), or 16,348 page-balanced rows (2*C*N over C CTA pairs: e.g.
 * C=32, N=128).
 *
 *   plan, q, latent_cache, num_blocks, block_table, seq_lens, softmax_scale,
 *   out, lse, stream   as for mla_decode.
 *   device_status      optional device int32[2] (4-byte aligned) that receives
 *                      the device-detected status (MLA_OK or MLA_ERR_*) and a
 *                      detail word; the call zeroes it first. Only these two
 *                      words are written. NULL keeps the status inside the
 *                      library's scratch, unreadable.
 *
 * Every call zeroes the array's status header (8 KiB, on `stream`) before its
 * kernels, so the counters a timed-out call left behind cannot mislead the
 * next one. The first call on each device looks up the array's device address
 * (with that device current) and caches it; make that first call before any
 * stream capture. Every call uses the same array and leaves its contents
 * behind, so calls that overlap on the GPU (other streams, other host
 * threads, the same device) race with each other: serialise them.
 */
int mla_decode_noalloc(const mla_decode_plan_t* plan, const void* q, const void* latent_cache,
                       int64_t num_blocks, const int32_t* block_table, const int32_t* seq_lens,
                       float softmax_scale, void* out, float* lse, int32_t* device_status,
                       void* stream);

/*
 * mla_merge_splits -- LSE-weighted merge of S partial attention results.
 *
 * vLLM names this merge_attn_states (mla_attention API docs, module docstring
 * "Chunked Prefill"; accumulate_mla_context_chunk) and uses it for the
 * decode-context-parallel combine as well. For each (b, h):
 *     M   = max_s lse_part[b,h,s]
 *     lse = M + ln sum_s exp(lse_part[b,h,s] - M)
 *     out = sum_s exp(lse_part[b,h,s] - lse) * o_part[b,h,s,:]
 * A partial with lse = -inf carries no weight; if all are -inf the result is
 * out = 0, lse = -inf (neutralize_empty_context_partials on the same page).
 *
 *   o_part     device, fp32 [B, N, S, v_dim], each partial already normalised.
 *   lse_part   device, fp32 [B, N, S], natural log.
 *   v_dim      a multiple of 8, 8 <= v_dim <= 2048.
 *   out        device, bf16 [B, N, v_dim].
 *   lse        device, fp32 [B, N], or NULL.
 * B * N above INT_MAX gives MLA_ERR_UNSUPPORTED.
 */
int mla_merge_splits(const float* o_part, const float* lse_part, int batch, int num_heads,
                     int num_splits, int v_dim, void* out, float* lse, void* stream);

/*
 * Uniform multi-token decode (vLLM mla_attention API docs,
 * QueryLenSupport.UNIFORM: every request has the same query length
 * q_len = T > 1, e.g. speculative decoding; MLACommonMetadataBuilder.build:
 * the query block is causal unless a non-causal one is allowed).
 *
 * The T new tokens are already in the cache, so request b holds
 * L = seq_lens[b] tokens and its query token i (0 <= i < T) sits at position
 * L - T + i. With `causal` != 0 it attends to tokens t <= L - T + i (a token
 * that sees none, when L < T - i, gets out = 0, lse = -inf); otherwise to all
 * t < L.
 *
 *   plan          one of two shapes, which selects how the work is laid out:
 *                 (a) T * N <= 128: mla_decode_plan with batch = B and
 *                     num_heads = T * N (the tokens' heads are the rows of
 *                     one decode, which reads each page once; host lengths,
 *                     if given, are the requests' lengths);
 *                 (b) mla_decode_plan with batch = B * T rows (row
 *                     r = b * T + i) of N heads and, if given, the host
 *                     lengths of those rows (the visible lengths above).
 *   num_heads     N, the heads of one query token.
 *   q             device, bf16 [B, T, N, 576] contiguous.
 *   block_table   device, int32 [B, max_blocks_per_seq]; seq_lens int32 [B].
 *   out, lse      device, bf16 [B, T, N, 512] and fp32 [B, T, N] (or NULL).
 *   workspace     as for mla_decode with this plan.
 *   scratch       shape (b) only (else may be NULL): device, >=
 *                 mla_multi_token_scratch_bytes(B, T, max_blocks_per_seq)
 *                 bytes, 256-byte aligned: the rows' block tables and lengths.
 * Shape (a) is one mla_decode launch (plus its merge); shape (b) one small
 * launch that writes the rows' block tables and lengths into `scratch`, then
 * mla_decode over the B * T rows (each row reads its request's pages).
 * Errors as mla_decode; a plan of neither shape or q_len < 1 gives
 * MLA_ERR_INVALID_ARG, scratch too small or misaligned MLA_ERR_WORKSPACE.
 */
size_t mla_multi_token_scratch_bytes(int batch, int q_len, int max_blocks_per_seq);

/*
 * mla_multi_token_row_lens -- host only, no device work: the number of cached
 * tokens each (request, query token) row sees, row r = b * q_len + i, under
 * the reading above: max(L - (q_len - 1 - i), 0) with `causal` != 0, else L
 * (L = seq_lens_host[b]). These are the host lengths a shape-(b) plan is made
 * from (mla_decode_plan with batch = B * q_len).
 *
 *   seq_lens_host   host, int32 [batch], every entry >= 0.
 *   row_lens_host   host, int32 [batch * q_len], written.
 * Returns MLA_ERR_INVALID_ARG for a null pointer, batch < 0, q_len < 1 or a
 * negative length (nothing written).
 */
int mla_multi_token_row_lens(const int32_t* seq_lens_host, int batch, int q_len, int causal,
                             int32_t* row_lens_host);
int mla_decode_multi_token(const mla_decode_plan_t* plan, int q_len, int num_heads, int causal,
                           const void* q, const void* latent_cache, int64_t num_blocks,
                           const int32_t* block_table, const int32_t* seq_lens,
                           float softmax_scale, void* out, float* lse, void* workspace,
                           size_t workspace_bytes, void* scratch, size_t scratch_bytes,
                           void* stream);

/*
 * Decode context parallelism (DCP): each of `world` ranks holds a shard of
 * every request's cached tokens, runs mla_decode over its shard (with its own
 * block table and the shard lengths below as seq_lens), and the ranks'
 * (out, lse) pairs, once gathered, are combined. vLLM mla_attention API docs,
 * MLAAttention.forward (forward_mqa per rank, then dcp_manager.combine with
 * the returned lse) and MLACommonMetadataBuilder (cp_kv_cache_interleave_size
 * as the local block, dcp_local_seq_lens as the rank's seq_lens).
 *
 * mla_dcp_local_seq_lens -- host only, no device work.
 * Token t of a request belongs to rank (t / interleave) % world, at index
 * (t / (interleave * world)) * interleave + t % interleave of that rank's
 * shard (runs of `interleave` tokens dealt round-robin). Writes, for every
 * request b, the number of its tokens that `rank` holds. Each shard length
 * is at most ceil(L / (world * interleave)) * interleave.
 *
 *   seq_lens_host   host, int32 [batch], every entry >= 0.
 *   world           >= 1; rank in [0, world); interleave >= 1.
 *   local_lens_host host, int32 [batch], written.
 * Returns MLA_ERR_INVALID_ARG for a null pointer, a negative length or
 * batch, or world / rank / interleave out of range (nothing written).
 */
int mla_dcp_local_seq_lens(const int32_t* seq_lens_host, int batch, int world, int rank,
                           int interleave, int32_t* local_lens_host);

/*
 * mla_dcp_combine -- combine the ranks' decode results, rank-major as an
 * all-gather over ranks leaves them:
 *     out_parts  device, bf16 [world, B, N, v_dim] (each rank's mla_decode out)
 *     lse_parts  device, fp32 [world, B, N] (each rank's mla_decode lse)
 * into out (bf16 [B, N, v_dim]) and lse (fp32 [B, N], or NULL) with the merge
 * identity of mla_merge_splits taken over the rank axis. A rank without
 * tokens of a request (out 0, lse -inf) carries no weight. Same argument
 * rules as mla_merge_splits (1 <= world <= 1024, v_dim a multiple of 8 in
 * [8, 2048]; out_parts and out 8-byte aligned); one kernel launch on
 * `stream`, no synchronisation.
 */
int mla_dcp_combine(const void* out_parts, const float* lse_parts, int world, int batch,
                    int num_heads, int v_dim, void* out, float* lse, void* stream);

/*
 * The steps on either side of the decode: per-head batched matmuls on the
 * tensor cores (vLLM mla_attention API docs, MLAAttention.forward_impl and
 * _v_up_proj; the weight layouts are the ones the raon-1-mini MLA page
 * prepares after loading: W_UK_T = W_UK.permute(1, 2, 0), W_UV transposed to
 * (N, Lkv, V)). Supported shapes: qk_nope_head_dim P = 128, RoPE width R = 64,
 * kv_lora_rank 512, v_head_dim 128, 1 <= num_heads <= 128, any batch.
 * Device-detected errors go to the status word of `workspace` (a status
 * header: device, >= 8192 bytes, 256-byte aligned, zeroed by
 * mla_workspace_init); read them with mla_read_error. One kernel launch on
 * `stream` each, no synchronisation. Every device pointer 16-byte aligned
 * (slot_mapping 8-byte aligned).
 *
 * mla_q_absorb_concat_cache -- the decode front end, in one launch
 * (raon-1-mini page, _decode_concat_cache: query concat fused with the
 * latent cache insert; RoPE is not applied here: q_pe and k_pe come in
 * already rotated):
 *     mqa_q[b, n, 0:512]   = sum_p q[b, n, p] * w_uk_t[n, p, 0:512]   (p < 128)
 *     mqa_q[b, n, 512:576] = q[b, n, 128:192]
 *     latent_cache row slot_mapping[b] = [kv_c[b, 0:512] | k_pe[b, 0:64]]
 *
 *   q             device, bf16 [B, N, 192] contiguous ([q_nope | q_pe]).
 *   w_uk_t        device, bf16 [N, 128, 512] contiguous.
 *   kv_c, k_pe    device, bf16 [B, 512] and [B, 64]: the new tokens' entries.
 *   slot_mapping  device, int64 [B]: row slot % 64 of block slot / 64 of
 *                 latent_cache (bf16 [num_blocks, 64, 576]); a negative slot
 *                 writes nothing (padding); a slot >= num_blocks * 64 is
 *                 recorded as MLA_ERR_BAD_BLOCK_ID (detail: slot / 64) and not
 *                 written. Non-negative slots must be distinct. NULL: no
 *                 insert (kv_c, k_pe, latent_cache unused).
 *   mqa_q         device, bf16 [B, N, 576], written (the decode's q).
 * Accumulation in fp32, one rounding to bf16 (nearest even).
 */
int mla_q_absorb_concat_cache(const void* q, const void* w_uk_t, const void* kv_c,
                              const void* k_pe, const int64_t* slot_mapping, void* latent_cache,
                              int64_t num_blocks, int batch, int num_heads, void* mqa_q,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * mla_v_up_proj -- the up-projection after the decode:
 *     out[b, n, 0:128] = sum_l x[b, n, l] * w_uv[n, l, 0:128]   (l < 512)
 *
 *   x     device, bf16 [B, N, 512] contiguous (mla_decode's out).
 *   w_uv  device, bf16 [N, 512, 128] contiguous.
 *   out   device, bf16 [B, N, 128] contiguous, written.
 * Accumulation in fp32, one rounding to bf16 (nearest even).
 */
int mla_v_up_proj(const void* x, const void* w_uv, int batch, int num_heads, void* out,
                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * mla_merge_splits_v_up_proj -- the split merge and the up-projection in one
 * launch: for every (b, n) the S partials are merged as mla_merge_splits does,
 * the merged row is rounded to bf16 (the precision of mla_decode's output)
 * and multiplied by W_UV[n] on the tensor cores without leaving the SM:
 *     x[b, n, :]   = bf16(sum_s exp(lse_part[b,n,s] - lse) * o_part[b,n,s,:])
 *     out[b, n, :] = sum_l x[b, n, l] * w_uv[n, l, 0:128]
 * (vLLM mla_attention API docs: the split partials' merge_attn_states, then
 * _v_up_proj; the weight layout is the raon-1-mini page's W_UV as (N, Lkv, V)).
 * The [B, N, 512] merged rows never go through HBM unless latent_out is given.
 *
 *   o_part, lse_part  device, fp32 [B, N, S, 512] and [B, N, S].
 *   num_splits        1 <= S <= 512 (more: MLA_ERR_UNSUPPORTED).
 *   w_uv              device, bf16 [N, 512, 128].
 *   out               device, bf16 [B, N, 128].
 *   lse, latent_out   device, fp32 [B, N] and bf16 [B, N, 512], each optional.
 *   workspace         a status header (>= 8192 bytes, 256-byte aligned).
 * One kernel launch on `stream`; every pointer 16-byte aligned (lse_part and
 * lse 4-byte).
 */
int mla_merge_splits_v_up_proj(const float* o_part, const float* lse_part, int batch,
                               int num_heads, int num_splits, const void* w_uv, void* out,
                               float* lse, void* latent_out, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * mla_decode_v_up_proj -- the decode followed by the up-projection: out[b, n, :]
 * = mla_decode's out[b, n, :] (bf16) times w_uv[n] (bf16 [N, 512, 128]),
 * i.e. forward_mqa then _v_up_proj of the vLLM mla_attention API docs. With a
 * split plan (S > 1, at most 512) the decode kernel's fp32 partials go
 * straight into mla_merge_splits_v_up_proj, and the latent rows are written
 * only if latent_out is given. Otherwise (S = 1 or the page-balanced
 * schedule) the decode writes latent_out (then required) and mla_v_up_proj
 * reads it back. Arguments as mla_decode, plus w_uv and out (bf16
 * [B, N, 128]); lse optional. Two launches (three with a page-balanced
 * merge), no synchronisation.
 */
int mla_decode_v_up_proj(const mla_decode_plan_t* plan, const void* q, const void* latent_cache,
                         int64_t num_blocks, const int32_t* block_table, const int32_t* seq_lens,
                         float softmax_scale, const void* w_uv, void* out, float* lse,
                         void* latent_out, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * mla_read_error -- synchronise `stream`, then read and clear the device
 * status word of `workspace`. *device_status receives MLA_OK or the first
 * MLA_ERR_* a kernel recorded since the last read. Returns MLA_ERR_CUDA if
 * the synchronisation or copy fails.
 */
int mla_read_error(void* workspace, int* device_status, void* stream);

/* Human-readable text for a status code (static storage). */
const char* mla_status_string(int status);

/* ABI version (MLA_DECODE_ABI_VERSION) of the loaded library. */
int mla_abi_version(void);

/*
 * mla_debug_gather_pages -- test hook for the page-table reading.
 *
 * Copies, for every request b and token t < seq_lens[b], the 576-wide cache
 * row of token t (row t % 64 of block block_table[b, t / 64]) into
 * dst[b, t, 0:576] (bf16 [B, dst_max_tokens, 576], contiguous) with plain
 * 16-byte loads and stores (no tensor map: the decode kernels' own loader is
 * checked by mla_debug_loader_pages). Rows t >= seq_lens[b] of dst are left
 * untouched. Block ids outside [0, num_blocks) are recorded in the workspace
 * status word and their rows are left untouched. This is the semantics of
 * vLLM's gather_cache / cp_gather_cache (mla_attention API docs,
 * _compute_prefill_context). `workspace` is a status header: device, >= 8192
 * bytes, 256-byte aligned, zeroed by mla_workspace_init.
 */
int mla_debug_gather_pages(const void* latent_cache, int64_t num_blocks,
                           const int32_t* block_table, const int32_t* seq_lens,
                           int batch, int max_blocks_per_seq, int dst_max_tokens,
                           void* dst, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * mla_debug_loader_pages -- test hook: the tensor-core decode kernel's own page
 * loaders, run alone.
 *
 * Launches the tensor-core decode kernel of `plan` (MLA_KERNEL_TC, any
 * schedule) in a mode where only its two TMA page loaders run: the same
 * segment walk over the plan's work, the same block-table reads, the same
 * tensor map over the cache viewed as [num_blocks * 64, 576] with 64 x 64
 * boxes at row block * 64, into the same swizzled shared-memory rings. Each
 * CTA then copies every page it received out of its rings: CTA rank r of a
 * pair writes the rows of token t of request b, as it holds them, to
 * dst[r, b, t, 0:576] (bf16 [2, B, dst_max_tokens, 576], contiguous). A CTA
 * receives all 576 columns of each page of its pair's work (its value
 * columns in one ring, the rest in the other), so both halves of dst hold
 * every token of every request whose pages the plan covers. Rows past a
 * request's length, or at t >= dst_max_tokens, are not written. Block ids
 * outside [0, num_blocks) are recorded (MLA_ERR_BAD_BLOCK_ID) and their rows
 * are written as zeros, which is what the decode reads there. No MMA runs and
 * q is not read. workspace: a status header as for mla_debug_gather_pages.
 * MLA_ERR_UNSUPPORTED for a plan of the CUDA-core kernel.
 */
int mla_debug_loader_pages(const mla_decode_plan_t* plan, const void* latent_cache,
                           int64_t num_blocks, const int32_t* block_table,
                           const int32_t* seq_lens, int dst_max_tokens, void* dst,
                           void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* MLA_DECODE_H */
