/*
 * mla_split_kv.h -- C ABI of the GB300 (sm_103a) MLA split-KV decode library.
 *
 * Matrix-absorbed MLA decode over a paged compressed-latent KV cache. Every
 * cached token holds a 512-wide latent `ckv` (the key *and* the value of
 * absorbed attention) and a 64-wide rotary key `kpe`. A decode call is
 *
 *     mla_plan            (host)   pick partitions per request, cut each
 *                                  request's tokens into block-aligned chunks
 *     mla_decode_partial  (device) one normalized fp32 partial + base-2 LSE
 *                                  per (chunk, query row, head)
 *     mla_merge_states    (device) LSE-weighted merge of a request's partials,
 *                                  rounded once to the output dtype
 *
 * Sources of the operation (web pages; cited by title and section):
 *  - "feat(core): matrix-absorbed MLA decode over a compressed-latent KV cache"
 *    (mlxcel PR #995), *What changed*: absorbed decode is
 *    SDPA(q_absorbed, ckv, ckv, scale, mask = scale * q_pe @ kpe^T + causal);
 *    Stage 2 cuts the latent range into chunks, each producing a normalized
 *    partial and its log2 LSE; *How #898's merge kernel is reused*: the merge
 *    contract H = num_heads, D = kv_lora_rank, M = batch, N = batch * chunks,
 *    o_indptr request-major, LSE in base 2.
 *  - "[kernel] Wire MLA split-KV decode" (vllm-metal PR #601), *What changed*:
 *    the decode kernel runs over a slice of the context; a reduce kernel
 *    combines slices by their LSE; host dispatch picks the split only for
 *    conservative cases (pure decode, long context, small launch, 2 to 8
 *    partitions, bounded temporary memory). Review: thresholds belong in a
 *    device-aware split-plan helper, and tests must assert the chosen plan.
 *  - MTPLX PR #639, commit log: segments of a non-contiguous history are
 *    attended separately and merged by LSE; a row with no visible key has
 *    LSE = -inf, weight 0 and merges to zeros; fp32 per-segment outputs are
 *    rounded once, after the merge; unsupported shapes bail without a launch.
 *
 * Conventions for every call:
 *  - All device buffers are caller-owned and stay owned by the caller. The
 *    library never allocates device memory in these calls and never
 *    synchronizes the stream; work is enqueued on `stream` (a cudaStream_t
 *    passed as void*, NULL = the legacy default stream).
 *  - Argument and shape errors are detected on the host and returned before
 *    anything is launched (the launch counters do not move).
 *  - Layouts are dense row-major with the innermost dimension last.
 *  - Supported: num_heads in {16, 64, 128}; kv_lora_rank 512; rope dim 64;
 *    block_size in {16, 32, 64}; q_len in [1, 32]; fp16 or bf16 inputs.
 *    Anything else returns MLA_ERR_UNSUPPORTED.
 */
#ifndef MLA_SPLIT_KV_H
#define MLA_SPLIT_KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_KV_LORA_RANK 512
#define MLA_ROPE_DIM 64
#define MLA_MAX_Q_LEN 32

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned buffer       */
  MLA_ERR_UNSUPPORTED = 2,  /* shape or dtype outside the supported set       */
  MLA_ERR_CUDA = 3,         /* a CUDA runtime/driver call or launch failed     */
  MLA_ERR_TIMEOUT = 4,      /* a bounded device-side wait ran out              */
  MLA_ERR_DEVICE_CHECK = 5, /* the device flagged bad data (e.g. page id)      */
  MLA_ERR_CAPACITY = 6      /* caller-provided plan arrays are too small       */
} mla_status_t;

/* MLA_E4M3: 8-bit E4M3 latent caches (sign, 4 exponent bits with bias 7, 3
 * mantissa bits; exponent field 0 subnormal; S.1111.111 NaN, no infinities)
 * read with a scalar cache scale, beside fp16 queries. */
typedef enum { MLA_F16 = 0, MLA_BF16 = 1, MLA_F32 = 2, MLA_E4M3 = 3 } mla_dtype_t;

/* Which partial-decode kernel runs. AUTO picks the tensor-core kernel. */
typedef enum {
  MLA_KERNEL_AUTO = 0,
  MLA_KERNEL_SIMT = 1,   /* CUDA-core fp32 FMA kernel                        */
  MLA_KERNEL_TC = 2      /* tcgen05/TMEM tensor-core kernel                  */
} mla_kernel_t;

/* One partition: logical tokens [t0, t1) of request b; its partial and LSE go
 * to row `out_slot` of the partials/lse buffers. */
typedef struct {
  int32_t b, t0, t1, out_slot;
} mla_chunk_t;

/* Device facts the planner sizes the launch by (mla_device_query fills it;
 * tests may fill it by hand). max_clusters[k] = co-resident clusters of 2^k
 * CTAs of the partial kernel (k = 0..4), 0 when that size cannot launch. */
typedef struct {
  int32_t num_sms;
  int32_t max_clusters[5];
} mla_device_info_t;

/*
 * mla_device_query -- fill *info for CUDA device `device` (-1 = current).
 * Returns MLA_ERR_CUDA when no device is usable.
 */
mla_status_t mla_device_query(int32_t device, mla_device_info_t* info);

#define MLA_MERGE_ENTRIES 0
#define MLA_MERGE_PARTIALS 1

/* mla_decode_desc_t.score_exchange */
#define MLA_SCORE_EXCHANGE_EXACT 0
#define MLA_SCORE_EXCHANGE_F16 1
#define MLA_SCORE_EXCHANGE_NONE 2
#define MLA_SCORE_EXCHANGE_F32 3

/* mla_decode_desc_t.decode_merge (see mla_decode) */
#define MLA_DECODE_MERGE_ENTRIES 0
#define MLA_DECODE_MERGE_TICKETS 1

/* Planner input/output. The caller sets the inputs and provides the host
 * arrays; mla_plan fills the outputs. */
typedef struct {
  /* inputs */
  int32_t max_partitions;   /* per-request cap; 0 = 8 (the pages' 2..8 gate)  */
  int32_t min_partitions;   /* floor for a request that is split; 0 = 2       */
  int32_t split_min_tokens; /* contexts shorter than this are not split;
                               0 = 4096                                        */
  int32_t dtype;            /* MLA_F16, MLA_BF16 or MLA_E4M3 (sets rows per CTA;
                               E4M3 caches need clusters of 2 or more)         */
  int32_t capacity;         /* entries available in `chunks`                   */
  mla_chunk_t* chunks;      /* host, caller-owned, >= capacity entries         */
  int32_t* o_indptr;        /* host, caller-owned, >= B+1 entries              */
  int32_t merge_path;       /* how the partitions will be merged, which sets
                               what spreading a partition over clusters costs:
                               MLA_MERGE_ENTRIES (0, default: mla_decode on
                               the paired kernel) or MLA_MERGE_PARTIALS
                               (mla_decode_partial + mla_merge_states, or
                               mla_decode's MLA_DECODE_MERGE_TICKETS way).
                               Other values:
                               INVALID_ARG.                                     */
  /* outputs */
  int32_t num_chunks;       /* N = sum_b P_b                                   */
  int32_t cluster_ctas;     /* CTAs per cluster (1,2,4,8,16)                    */
  int32_t kernel;           /* mla_kernel_t the plan was sized for             */
  int32_t clusters_per_chunk; /* k >= 1 clusters share one partition; k > 1
                               needs a workspace (mla_workspace_bytes)         */
} mla_plan_t;

/*
 * mla_plan -- choose P_b partitions per request and cut [0, L_b) into P_b
 * contiguous block-aligned chunks (vllm-metal PR #601 *What changed*: host
 * dispatch picks the split; mlxcel PR #995 `MlaSplitPlan` cuts the latent
 * range). Chunk p of request b covers [min(p*C, L), min((p+1)*C, L)) with
 * C = ceil(ceil(L/P)/bs)*bs. Chunks are emitted request-major, out_slot = the
 * chunk's index, o_indptr[b] = first chunk of request b, o_indptr[B] = N.
 *
 * Rule (device-aware): a request shorter than split_min_tokens gets P = 1;
 * otherwise P_b is proportional to L_b so that all partitions fill one wave
 * of the device's co-resident clusters, clamped to [min, max] partitions and
 * so that no chunk is empty. cluster_ctas is the cluster size that keeps the
 * most CTAs busy in that wave with at least one 64-token tile per CTA; when
 * the paired 16-row kernel applies (q_len*H <= 16) and the device has CTA
 * pairs, clusters of one are not considered. When the paired 16-row kernel
 * applies (q_len*H <= 16, clusters of >= 2)
 * and one wave holds more clusters than partitions, each partition is spread
 * over clusters_per_chunk = k clusters (k <= 16, every CTA pair keeping at
 * least one 128-token tile); the partition count itself is not raised. For a
 * single long request on that kernel, P, the cluster size and k are chosen
 * by a time model among the plans whose P * k clusters are all co-resident
 * (one wave): 1.75 us per 128-token tile of the busiest CTA pair (a chunk's
 * tiles split evenly over its k * cluster/2 pairs), plus 0.6 us per further
 * round of 96 entries in the entries merge when the parts are merged as pair
 * entries (merge_path MLA_MERGE_ENTRIES: a spread costs nothing more), or,
 * for k > 1, 6 us + 0.3 us x 2k / cluster when each chunk's parts are first
 * merged into its partial (MLA_MERGE_PARTIALS); on a tie, more CTA pairs, then
 * fewer clusters per partition. Constants fitted to steady-state layer-call
 * times measured on GB300.
 *
 * context_lens_host: host [B] int32, each >= 0. dev: from mla_device_query or
 * hand-filled. Returns MLA_ERR_CAPACITY when N > plan->capacity (num_chunks
 * then holds the size needed), MLA_ERR_INVALID_ARG / MLA_ERR_UNSUPPORTED for
 * bad arguments. Pure host code; touches no GPU.
 */
mla_status_t mla_plan(const int32_t* context_lens_host, int32_t B, int32_t num_heads,
                      int32_t q_len, int32_t block_size, const mla_device_info_t* dev,
                      mla_plan_t* plan);

/* Shapes and launch options of mla_decode_partial. */
typedef struct {
  int32_t num_requests;       /* B                                            */
  int32_t num_heads;          /* H in {16, 64, 128}                           */
  int32_t q_len;              /* query rows per request, 1..32                */
  int32_t block_size;         /* tokens per page: 16, 32 or 64                */
  int32_t num_blocks;         /* pages in the cache pool                      */
  int32_t max_blocks_per_req; /* row stride of block_table, in entries        */
  int32_t dtype;              /* MLA_F16 or MLA_BF16 (q, ckv, kpe), or MLA_E4M3:
                                 ckv and kpe 8-bit E4M3 (576 bytes a token),
                                 q fp16; E4M3 runs on the CTA-pair kernels
                                 only (q_len * H <= 16: clusters of 2..16 CTAs;
                                 more rows: clusters of 2 (or 0 = auto); not
                                 MLA_KERNEL_SIMT), else UNSUPPORTED            */
  int32_t causal;             /* 1: the q_len rows are the last q_len tokens
                                 of each request; row i sees t <= L-q_len+i    */
  const mla_chunk_t* chunks;  /* DEVICE array of num_chunks records, or NULL
                                 for a uniform split into num_partitions       */
  int32_t num_chunks;         /* records in `chunks` (ignored when NULL)      */
  int32_t cluster_ctas;       /* CTAs per cluster: 1,2,4,8,16; 0 = auto       */
  int32_t kernel;             /* mla_kernel_t                                 */
  void* stream;               /* cudaStream_t                                 */
  int32_t clusters_per_chunk; /* k: clusters per partition; 0 or 1 = one.
                                 k > 1 (1..16): the chunk's tokens are split
                                 over k clusters; each CTA pair writes its part
                                 (unnormalized O, row maxima and sums) to the
                                 workspace and the CTA that finishes last
                                 merges them in index order into the
                                 partition's slot. Only for the 16-row
                                 tensor-core kernel whose CTAs share tiles in
                                 pairs (q_len*H <= 16, cluster_ctas set to
                                 2..16, not 0 = auto);
                                 otherwise MLA_ERR_UNSUPPORTED (INVALID_ARG for
                                 cluster_ctas 0 or a missing / short workspace;
                                 k > 16 is INVALID_ARG).                         */
  void* workspace;            /* DEVICE, >= mla_workspace_bytes(...) bytes,
                                 16-byte aligned, ZEROED by the caller before
                                 its first use; every call leaves its counters
                                 at zero again (after a device error, zero it
                                 again). Calls sharing a workspace must not
                                 overlap in time. Unused when k <= 1.           */
  uint64_t workspace_bytes;   /* size of `workspace`                          */
  int32_t tables_ready;       /* 1: `chunks`, context_lens and block_table
                                 (and mla_decode's o_indptr) are complete
                                 before the kernel that precedes this call in
                                 the stream starts (for instance copied from
                                 the host before the decode step); the paired
                                 16-row kernel and the entries merge kernel,
                                 programmatic dependent launches, then read
                                 them while the kernel before them finishes
                                 instead of after it. Queries are always read
                                 after it, caches too unless prefix_ready. 0
                                 (default): every input is read after the
                                 preceding kernel has finished. Other values:
                                 INVALID_ARG.                                  */
  int32_t decode_merge;       /* mla_decode only, how the paired 16-row kernel's
                                 parts reach `out`: MLA_DECODE_MERGE_ENTRIES
                                 (0, default) or MLA_DECODE_MERGE_TICKETS (1),
                                 see mla_decode. Other values: INVALID_ARG.
                                 mla_decode_partial ignores it.                */
  int32_t prefix_ready;       /* 1 (needs tables_ready = 1): the cache rows of
                                 every position before each request's window
                                 (positions < context_len - q_len) are final
                                 before the kernel that precedes this call in
                                 the stream ends (that kernel may write the
                                 window's rows, as mla_cache_append of this
                                 call's new tokens does). The paired 16-row
                                 kernel then loads its first tiles (one per
                                 tile slot) that lie wholly before the window
                                 while that kernel finishes; results are the
                                 same bits. Other kernels ignore it. 0
                                 (default): caches are read after it. Other
                                 values, or 1 with tables_ready = 0:
                                 INVALID_ARG.                                  */
  float cache_scale;          /* MLA_E4M3 caches: the value of a cache byte x is
                                 e4m3(x) * cache_scale, cache_scale in
                                 [2^-24, 2^24] (the scalar folded in as mlxcel
                                 PR #995, *What changed*, folds a global
                                 scale). It multiplies the score scale and the
                                 output: one fp32 rounding each, none for a
                                 power of two. Other dtypes: ignored. Anything
                                 else (0, negative, NaN, out of range) with
                                 E4M3: INVALID_ARG.                            */
  int32_t score_exchange;     /* the 128-row kernel (more than 16 rows): what
                                 the two CTAs of a pair send each other of
                                 their scores. MLA_SCORE_EXCHANGE_EXACT (0,
                                 default): exact; on 16-bit caches with at
                                 least 128 rows nothing crosses (as NONE),
                                 otherwise (64 rows, E4M3 caches) fp32
                                 partial scores of the real rows (as F32).
                                 MLA_SCORE_EXCHANGE_F16 (1): each CTA's partial
                                 dot product of a tile is rounded once to fp16
                                 (both CTAs add the same rounded values, so
                                 they still agree), halving the bytes that
                                 cross distributed shared memory; the error
                                 this adds grows with the scores' magnitude
                                 (|s| x 2^-12 per half, before the softmax
                                 scale), so it is a caller's choice.
                                 MLA_SCORE_EXCHANGE_NONE (2, 16-bit caches;
                                 E4M3: UNSUPPORTED): each CTA computes the full
                                 scores itself (part of the queries held in
                                 tensor memory, two full-width tile slots).
                                 MLA_SCORE_EXCHANGE_F32 (3): each CTA computes
                                 the scores over its half of the columns and
                                 the fp32 partial scores cross. The exact ways
                                 differ only in the order of fp32 sums. Other
                                 kernels ignore it. Other values: INVALID_ARG. */
} mla_decode_desc_t;

/*
 * mla_workspace_bytes -- device bytes a mla_decode_partial call with
 * clusters_per_chunk = k > 1 on clusters of cluster_ctas CTAs needs: two
 * uint32 tickets per chunk (256-byte aligned block), then E = N*k*cluster_ctas/2
 * entries (one per CTA pair of a chunk) of [q_len, H, 512] fp32, then E x 2
 * blocks of [q_len, H, 2] fp32 (each pair's row maxima and sums, one copy per
 * column half). 0 when k <= 1 or cluster_ctas < 2. No counterpart on the
 * pages: the split of a partition over several clusters is this library's way
 * to fill the GPU at the pages' 2..8 partitions.
 */
uint64_t mla_workspace_bytes(int32_t num_chunks, int32_t clusters_per_chunk, int32_t cluster_ctas, int32_t q_len,
                             int32_t num_heads);

/* Size of the library's own scratch used by mla_decode_partial_static. */
#define MLA_STATIC_WORKSPACE_BYTES (4u * 1024u * 1024u)

/*
 * mla_decode_partial_static -- mla_decode_partial for callers that cannot
 * provide a workspace: the same arguments and results, but a partition
 * spread over clusters (desc->clusters_per_chunk > 1) uses a scratch buffer
 * that lives in the library itself (a statically sized device array of
 * MLA_STATIC_WORKSPACE_BYTES bytes per device) instead of desc->workspace,
 * which is ignored. The call allocates nothing. The pages have no
 * counterpart: they split a partition over one thread group and need no
 * scratch.
 *
 * Set-up happens on the first call for a device (with that device
 * current): the scratch address is looked up and the scratch is cleared,
 * synchronously. Make that first call before any stream capture. The set-up
 * is kept for the life of the process: after cudaDeviceReset (or anything
 * else that replaces the device's primary context) this entry point must not
 * be used again in that process. Calls on one device share the scratch:
 * calls that may overlap in time (other streams, other threads) race and
 * give undefined results; calls in one stream are fine. Every call that
 * completes leaves the scratch's tickets at zero; a call stopped by a device
 * error may not, so mla_check_device_errors clears the current device's
 * scratch again whenever it finds the error word set.
 *
 * Returns MLA_ERR_CAPACITY (before any launch) when the call's spread plan
 * needs more than MLA_STATIC_WORKSPACE_BYTES (mla_workspace_bytes(...) of
 * the call), MLA_ERR_CUDA when the set-up fails, otherwise what
 * mla_decode_partial returns for the same descriptor without a workspace
 * (so an invalid or unsupported spread gets the same status from both).
 * With clusters_per_chunk <= 1 it is mla_decode_partial.
 */
mla_status_t mla_decode_partial_static(const void* q_absorbed, const void* q_pe, const void* ckv_cache,
                                       const void* kpe_cache, const int32_t* block_table,
                                       const int32_t* context_lens, float scale, int32_t num_partitions,
                                       float* partials, float* lse, const mla_decode_desc_t* desc);

/*
 * mla_decode_partial -- attention of every query row over one chunk of its
 * request's cached tokens, as a normalized partial and a base-2 LSE
 * (mlxcel PR #995 *What changed*, `mla/decode.rs` and `mla/split_kv.rs`;
 * vllm-metal PR #601 *What changed*, slice-capable `paged_mla_attention`).
 *
 * For request b, query row i (0 <= i < q_len), head h and chunk [t0, t1):
 *   s_t   = scale * (q_absorbed[b,i,h,:] . ckv[t,:]) + scale * (q_pe[b,i,h,:] . kpe[t,:])
 *           over the visible tokens t in [t0, t1) (all of them, or
 *           t <= L_b - q_len + i when causal)
 *   partial[slot,i,h,:] = sum_t softmax(s)_t * ckv[t,:]      (fp32)
 *   lse[slot,i,h]       = log2 sum_t exp(s_t)                (fp32)
 * An empty chunk (or a row with no visible token) gives partial = 0 and
 * lse = -inf. The token t of request b lives in cache row
 * block_table[b, t / bs] * bs + t % bs.
 *
 * q_absorbed : device [B, q_len, H, 512] dtype (fp16 for MLA_E4M3), 16-byte
 *              aligned
 * q_pe       : device [B, q_len, H, 64]  dtype (fp16 for MLA_E4M3), 16-byte
 *              aligned
 * ckv_cache  : device [num_blocks, bs, 512] dtype (bytes for MLA_E4M3),
 *              16-byte aligned
 * kpe_cache  : device [num_blocks, bs, 64]  dtype (bytes for MLA_E4M3),
 *              16-byte aligned
 * block_table: device [B, max_blocks_per_req] int32; entries past a request's
 *              last page are never read. An entry outside [0, num_blocks)
 *              reads zeros and raises MLA_ERR_DEVICE_CHECK at the next
 *              mla_check_device_errors.
 * context_lens: device [B] int32
 * scale      : softmax scale applied to both score terms
 * num_partitions: with desc->chunks == NULL, every request is split into this
 *              many chunks by the planner's chunk rule and chunk n = b*P + p
 *              writes slot n; ignored otherwise.
 * partials   : device [num_slots, q_len, H, 512] fp32 (written)
 * lse        : device [num_slots, q_len, H] fp32 (written)
 * Returns MLA_OK once the kernel is enqueued.
 */
mla_status_t mla_decode_partial(const void* q_absorbed, const void* q_pe, const void* ckv_cache,
                                const void* kpe_cache, const int32_t* block_table,
                                const int32_t* context_lens, float scale, int32_t num_partitions,
                                float* partials, float* lse, const mla_decode_desc_t* desc);

/*
 * mla_merge_states -- merge each request's partials by their base-2 LSE
 * (mlxcel PR #995 *How #898's merge kernel is reused*: the contract of
 * paged_attention_merge_states; vllm-metal PR #601: paged_mla_attention_reduce;
 * MTPLX PR #639: -inf rows and a single rounding after the merge).
 *
 * For request b (partials o_indptr[b] .. o_indptr[b+1]-1), row i, head h:
 *   M = max_p lse_p; if M = -inf: out = 0, out_lse = -inf;
 *   else w_p = 2^(lse_p - M), out = sum_p w_p partial_p / sum_p w_p,
 *        out_lse = M + log2 sum_p w_p.
 * The sum runs in fixed p order (bitwise reproducible) and `out` is rounded
 * once, to nearest-even, to out_dtype.
 *
 * partials : device [N, q_len, H, 512] fp32;  lse: device [N, q_len, H] fp32
 * o_indptr : device [B+1] int32, non-decreasing, o_indptr[0] = 0, and
 *            o_indptr[B] <= the slots held by partials / lse. The offsets are
 *            device data and are not checked: a table that breaks this reads
 *            outside the buffers (mla_plan's o_indptr always satisfies it).
 * out      : device [B, q_len, H, 512] of out_dtype (MLA_F16/BF16/F32)
 * out_lse  : device [B, q_len, H] fp32, or NULL
 */
mla_status_t mla_merge_states(const float* partials, const float* lse, const int32_t* o_indptr,
                              int32_t B, int32_t q_len, int32_t num_heads, void* out,
                              int32_t out_dtype, float* out_lse, void* stream);

/*
 * mla_decode -- one whole decode layer call: the attention of mla_decode_partial
 * merged as mla_merge_states merges it, over the request-major offsets o_indptr,
 * into `out` (rounded once to out_dtype) and `out_lse` (NULL allowed).
 *
 * The ways, by kernel and desc->decode_merge:
 *  - the paired 16-row kernel (q_len*H <= 16, clusters of 2..16 CTAs) with
 *    MLA_DECODE_MERGE_ENTRIES (default): the partial kernel skips its
 *    in-cluster combine and writes every CTA pair's unnormalized part (O over
 *    its tokens, row maxima and sums) to the workspace; a merge kernel launched
 *    as its programmatic dependent combines all the parts of a request
 *    straight into `out` (the merge of the pages' contract, M = max, weights
 *    2^(m - M), applied to the parts; the same bits on every call for the same
 *    plan). Its CTAs fit on an SM beside the partial kernel's, so it is
 *    resident before the partial kernel ends; it releases its own dependent at
 *    once (every kernel of this library waits for the kernel before it to
 *    complete before reading anything). `partials` and `lse` are not written.
 *  - the paired kernel with MLA_DECODE_MERGE_TICKETS: ONE launch that writes
 *    the chunk partials. "[kernel] Wire MLA split-KV decode" (vllm-metal PR
 *    #601), *What changed*, avoids a temporary by letting partition 0 write
 *    straight into the output; here the reduce moves into the partial kernel:
 *    once a chunk's partial is written (to partials / lse, as
 *    mla_decode_partial writes it), an acquire-release ticket per (request,
 *    column slice) counts it, and the CTA that counts a request's last chunk
 *    merges that slice of all the request's partials into `out` with the merge
 *    kernel's arithmetic in its order: the same bits as mla_decode_partial +
 *    mla_merge_states. Measured on GB300 it is slower than the default (the
 *    last CTAs do the whole merge); kept as an option.
 *  - other kernels: mla_decode_partial, then mla_merge_states, on `stream`
 *    (partials / lse written as those calls write them).
 *
 * o_indptr : device [B+1] int32, as for mla_merge_states; the chunks must be
 *            request-major with chunk n writing slot n, so that request b's
 *            chunks are exactly o_indptr[b] .. o_indptr[b+1]-1, and every request
 *            needs at least one chunk (mla_plan's tables do; with
 *            desc->chunks == NULL, o_indptr[b] = b * num_partitions). Device
 *            data: not checked.
 * out      : device [B, q_len, H, 512] of out_dtype (MLA_F16/BF16/F32)
 * out_lse  : device [B, q_len, H] fp32, or NULL
 * partials, lse: device, as for mla_decode_partial (scratch on the default path
 *            of the paired kernel)
 * desc->workspace: on the paired kernel DEVICE, >= mla_decode_workspace_bytes(...)
 *            bytes, 16-byte aligned, ZEROED by the caller before its first use;
 *            every completed call leaves its counters zeroed again (after a device
 *            error, zero it again). Other kernels: what mla_decode_partial needs.
 *            Calls sharing a workspace must not overlap in time.
 * Returns what mla_decode_partial and mla_merge_states return (and
 * MLA_ERR_INVALID_ARG for a NULL or misaligned o_indptr / out / out_lse, a
 * short workspace or a bad decode_merge value, MLA_ERR_UNSUPPORTED for another
 * out_dtype). No counterpart on the pages as one call: the pages launch a
 * partial kernel and a reduce kernel.
 */
mla_status_t mla_decode(const void* q_absorbed, const void* q_pe, const void* ckv_cache, const void* kpe_cache,
                        const int32_t* block_table, const int32_t* context_lens, float scale, int32_t num_partitions,
                        float* partials, float* lse, const int32_t* o_indptr, void* out, int32_t out_dtype,
                        float* out_lse, const mla_decode_desc_t* desc);

/* Workspace bytes of mla_decode on the paired kernel, one layout for both of
 * its ways: B * 16 uint32 request tickets and num_chunks * q_len * H fp32 LSE
 * copies (the TICKETS way's; each block 256-byte aligned), then two uint32
 * tickets per chunk (a 256-byte block; the TICKETS way's spread plans), then
 * E = num_chunks * max(1, clusters_per_chunk) * cluster_ctas / 2 entries (one
 * per CTA pair) of [q_len, H, 512] fp32 and E x [2, q_len, H, 2] fp32 row
 * maxima and sums. The default way writes only the entries, never a ticket,
 * so one zeroed workspace serves both ways in any order. */
uint64_t mla_decode_workspace_bytes(int32_t num_requests, int32_t num_chunks, int32_t clusters_per_chunk,
                                    int32_t cluster_ctas, int32_t q_len, int32_t num_heads);

/*
 * mla_cache_append -- write each request's newest tokens into the paged
 * cache, the step before attention in a decode layer call ("[kernel] Wire MLA
 * split-KV decode", *Bench*: the wrapper's cache write). Token i of the q_len
 * new tokens of request b goes to logical position t = context_lens[b] -
 * q_len + i (context_lens already counts the new tokens, as with a causal
 * window: its rows are the last q_len tokens), cache row
 * block_table[b, t / bs] * bs + t % bs. Positions t < 0 are not written. A
 * page outside the table row or the pool is not written and raises
 * MLA_ERR_DEVICE_CHECK at the next mla_check_device_errors.
 *
 * ckv_new  : device [B, q_len, 512] 16-bit (the caches' dtype), 16-byte aligned
 * kpe_new  : device [B, q_len, 64]  16-bit, 16-byte aligned
 * block_table, context_lens: as for mla_decode_partial
 * ckv_cache, kpe_cache: device, as for mla_decode_partial (written)
 * Returns MLA_OK once the copy kernel is enqueued. A programmatic dependent
 * launch: it waits for the kernel before it in the stream to complete before
 * reading anything, and lets the kernel after it start at once (every kernel
 * of this library waits for it before reading what it writes; with
 * prefix_ready the decode reads only rows before the window early).
 */
mla_status_t mla_cache_append(const void* ckv_new, const void* kpe_new, const int32_t* block_table,
                              const int32_t* context_lens, int32_t B, int32_t q_len, int32_t block_size,
                              int32_t num_blocks, int32_t max_blocks_per_req, void* ckv_cache, void* kpe_cache,
                              void* stream);

/*
 * mla_merge_unembed -- mla_merge_states followed by the output side of the
 * fold, the step after attention ("feat(core): matrix-absorbed MLA decode over
 * a compressed-latent KV cache", *What changed*: W_UV^T [1, H, r, v_head];
 * "[kernel] Wire MLA split-KV decode", *Bench*: the wrapper's unembed):
 *   out_v[b, i, h, :] = merged[b, i, h, :] @ W_UV^T[h]
 * where merged is what mla_merge_states computes in fp32 (the same bits; it
 * is never rounded here), the product accumulates in fp32 in a fixed order
 * (d in eight chunks of 64, each in order, the chunk sums added in order),
 * and the result is rounded once to out_dtype. out_lse (NULL allowed)
 * receives the merged LSE.
 *
 * w_uv_t : device [H, 512, v_head] of w_dtype (MLA_F16 / MLA_BF16), 16-byte
 *          aligned; v_head a multiple of 32, at most 512
 * out    : device [B, q_len, H, v_head] of out_dtype (MLA_F16 / BF16 / F32)
 * partials, lse, o_indptr: as for mla_merge_states
 * A programmatic dependent launch, like mla_merge_states; w_uv_t (a weight) is
 * read while the kernel before it in the stream finishes, so that kernel must
 * not write it.
 */
mla_status_t mla_merge_unembed(const float* partials, const float* lse, const int32_t* o_indptr, int32_t B,
                               int32_t q_len, int32_t num_heads, const void* w_uv_t, int32_t w_dtype, int32_t v_head,
                               void* out, int32_t out_dtype, float* out_lse, void* stream);

/*
 * mla_decode_unembed -- a layer call's attention with the unembed after it:
 * mla_decode's merged latent taken to the value space,
 *   out_v[b, i, h, :] = merged[b, i, h, :] @ W_UV^T[h]
 * ("feat(core): matrix-absorbed MLA decode over a compressed-latent KV cache",
 * *What changed*: the output side of the fold, W_UV^T [1, H, r, v_head];
 * "[kernel] Wire MLA split-KV decode", *Bench*: the wrapper unembeds the
 * attention output).
 *  - the paired kernel: every CTA pair writes its part to desc->workspace as
 *    mla_decode does, then ONE programmatic dependent launch merges a
 *    request's parts in the entries merge's arithmetic and order (its fp32
 *    latent is the bits mla_decode writes with MLA_F32, never rounded here)
 *    and takes the product with W_UV^T as mla_merge_unembed does. Only the
 *    default way: MLA_ERR_UNSUPPORTED for MLA_DECODE_MERGE_TICKETS.
 *  - other kernels: mla_decode_partial, then mla_merge_unembed.
 * Arguments: those of mla_decode (o_indptr, partials, lse and desc alike,
 * desc->workspace included), with w_uv_t, w_dtype, v_head, out_v and
 * out_dtype as for mla_merge_unembed (out_v: device [B, q_len, H, v_head]);
 * out_lse (NULL allowed) receives the merged LSE. Returns what mla_decode and
 * mla_merge_unembed return for the same arguments.
 */
mla_status_t mla_decode_unembed(const void* q_absorbed, const void* q_pe, const void* ckv_cache, const void* kpe_cache,
                                const int32_t* block_table, const int32_t* context_lens, float scale,
                                int32_t num_partitions, float* partials, float* lse, const int32_t* o_indptr,
                                const void* w_uv_t, int32_t w_dtype, int32_t v_head, void* out_v, int32_t out_dtype,
                                float* out_lse, const mla_decode_desc_t* desc);

/*
 * mla_check_device_errors -- synchronize `stream`, read and clear the device
 * error word the kernels set (bit 0: a bounded wait timed out; bit 1: a page
 * id outside the pool; bit 2: a kernel found its launch unusable -- the
 * paired kernel's shared memory not 1024-byte aligned -- and did nothing).
 * *code_out (nullable) receives the raw word. When the word was set it also
 * zeroes the current device's mla_decode_partial_static scratch (if set up),
 * since a call that stopped early may have left its tickets counted; a
 * caller-owned workspace must be zeroed again by its owner. Returns MLA_OK
 * when the word was 0, MLA_ERR_TIMEOUT or MLA_ERR_DEVICE_CHECK otherwise
 * (MLA_ERR_CUDA if a CUDA call fails).
 */
mla_status_t mla_check_device_errors(void* stream, uint32_t* code_out);

/*
 * mla_selfcheck -- run mla_plan, mla_decode_partial and mla_merge_states on
 * the current device over a built-in case whose answer is known in closed
 * form, and compare. The case has 2 requests (6000 and 700 tokens, ragged last
 * pages, pages of 32 tokens scattered over a 256-page pool whose unowned pages
 * hold 1000.0) and 16 heads: 15 heads whose query picks out one "needle"
 * token through either the rope key or one latent column (score 64 against
 * at most 16 elsewhere, so the merged output is that token's latent row and
 * the LSE is 64 log2 e), and one head with all-zero queries (the mean of the
 * latent rows, LSE log2 L; softmax of equal scores, mlxcel PR #995 *What
 * changed*: the partial is normalized, the LSE in base 2). It runs in fp16
 * and bf16, on the planner's default kernel choice and on the CUDA-core
 * kernel.
 *
 * Unlike the other calls it allocates device memory (about 25 MB), creates
 * and synchronizes its own stream, and reads and clears the device error
 * word (as mla_check_device_errors does). Not for a hot path.
 * *max_abs_err (nullable) receives the largest |output - expected| seen.
 * Returns MLA_OK when every output row is within 1e-6 (needle rows, exact in
 * fp32) or 2e-3 (the mean row) and every LSE within 1e-3;
 * MLA_ERR_DEVICE_CHECK on a mismatch; otherwise the first failing call's
 * status (MLA_ERR_CUDA without a usable device).
 */
mla_status_t mla_selfcheck(float* max_abs_err);

/* Launch counters proving which kernel ran (mlxcel PR #995 `mla/stats.rs`:
 * per-path counters read around a measured region). Indices: */
#define MLA_CTR_PARTIAL_SIMT 0
#define MLA_CTR_PARTIAL_TC 1
#define MLA_CTR_MERGE 2
#define MLA_CTR_REJECTED 3
#define MLA_CTR_CTAS 4 /* CTAs launched by partial kernels */
#define MLA_CTR_DECODE_FUSED 5 /* mla_decode calls that ran as one launch */
#define MLA_CTR_WRAP 6 /* mla_cache_append, mla_merge_unembed and mla_decode_unembed unembed launches */
#define MLA_NUM_COUNTERS 7
/* mla_get_counters -- copy min(n, MLA_NUM_COUNTERS) counters to out (host). */
void mla_get_counters(uint64_t* out, int32_t n);
void mla_reset_counters(void);

/* The bounded device waits give up after this many nanoseconds (default
 * 2e9), flag MLA_ERR_TIMEOUT and let the kernel exit. Host state; applies to
 * launches issued after the call. */
void mla_set_wait_timeout_ns(uint64_t ns);

/* Bytes of the partials and lse buffers for N slots. */
size_t mla_partials_bytes(int32_t num_slots, int32_t q_len, int32_t num_heads);
size_t mla_lse_bytes(int32_t num_slots, int32_t q_len, int32_t num_heads);

const char* mla_status_string(mla_status_t status);
int32_t mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_SPLIT_KV_H */
