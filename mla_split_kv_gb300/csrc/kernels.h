// Internal interface between the C-ABI layer and the kernels (not installed).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mla {

constexpr int kRank = 512;        // kv_lora_rank: width of ckv
constexpr int kRope = 64;         // rope dim: width of kpe
constexpr int kQkDim = kRank + kRope;
constexpr int kTileTokens = 64;   // tokens per pipeline tile
constexpr int kBoxCols = 64;      // 16-bit columns per TMA box (128 bytes)
constexpr int kBoxesPerTile = kQkDim / kBoxCols;  // 8 ckv boxes + 1 kpe box
constexpr int kBoxBytes = kTileTokens * kBoxCols * 2;  // 8 KB
constexpr int kTileBytes = kBoxesPerTile * kBoxBytes;  // 72 KB

// Device error bits (the per-file g_device_error words).
constexpr uint32_t MLA_DEVERR_TIMEOUT = 1u;
constexpr uint32_t MLA_DEVERR_BAD_PAGE = 2u;
constexpr uint32_t MLA_DEVERR_CONFIG = 4u;  // a kernel found its launch unusable (shared memory alignment)

struct PartialParams {
  const uint16_t* q_abs;       // [B, q_len, H, 512]
  const uint16_t* q_pe;        // [B, q_len, H, 64]
  const int32_t* block_table;  // [B, max_blocks]
  const int32_t* context_lens; // [B]
  const uint8_t* ckv;          // ckv cache base: page g at g * bs * 1024 bytes
  const uint8_t* kpe;          // kpe cache base: page g at g * bs * 128 bytes
  const void* chunks;          // device int4 {b, t0, t1, slot} per chunk, or null
  float* partials;             // [slots, q_len, H, 512]
  float* lse;                  // [slots, q_len, H]
  float scale_log2;            // softmax scale * log2(e)
  int32_t B, H, q_len, bs, max_blocks, num_blocks;
  int32_t num_parts;           // uniform split when chunks == null
  int32_t causal;
  int32_t tables_ready;        // chunks / context_lens / block_table may be read before the dependency wait
  int32_t fp8;                 // E4M3 caches (the paired kernel): loaded as bytes, converted to fp16 in the slot
  float cache_scale;           // E4M3: the value of byte x is e4m3(x) * cache_scale (folded into scale_log2 and O)
  int32_t prefix_ready;        // cache rows before each request's window may be read before the dependency wait
  int32_t xchg16;              // the 128-row kernel: 1 partial scores cross the pair as fp16, 2 none cross
  uint64_t timeout_ns;
  // a chunk spread over `subs` clusters (the paired 16-row kernel): grid.y = chunks * subs.
  // One entry per CTA pair of a chunk (subs * cluster / 2 of them): its unnormalized O^T in
  // ws_partials and its row maxima / sums in ws_lse; two tickets per chunk (one per column
  // half). Tickets are zero between calls.
  int32_t subs;
  float* ws_partials;          // [entries, q_len, H, 512]
  float* ws_lse;               // [entries, 2, q_len, H, 2]
  uint32_t* ws_tickets;        // [chunks, 2]
  // Single-launch decode (out != null): once a request's chunk partials are written, the CTA
  // that finishes last for a column slice of the request merges that slice of all of them into
  // `out`, with the merge kernel's arithmetic. Tickets: [B][kSliceTickets], zero between calls.
  // lse_copy: [slots, q_len, H], the second column half's copy of each chunk's LSE (spread plans).
  const int32_t* o_indptr;     // [B+1] request-major chunk offsets (device)
  void* out;                   // [B, q_len, H, 512] of out_dtype, or null
  float* out_lse;              // [B, q_len, H], or null
  int32_t out_dtype;           // MLA_F16 / MLA_BF16 / MLA_F32
  uint32_t* req_tickets;
  float* lse_copy;
  // the paired kernel writes every CTA pair's part (unnormalized O^T, row maxima and sums) as an
  // entry of ws_partials / ws_lse and nothing else; the entries merge kernel combines them
  int32_t entries_only;
};
constexpr int kSliceTickets = 16;  // per request: one per column slice (cluster rank) or column half

// The merge of the paired kernel's pair entries (entries_only): request b's entries are
// [o_indptr[b] * epc, o_indptr[b+1] * epc), epc = entries per chunk.
struct EntryMergeParams {
  const float* ws_partials;    // [entries, rows, 512] unnormalized O
  const float* ws_lse;         // [entries, 2, rows, 2] row maximum and sum (two equal copies)
  const int32_t* o_indptr;     // [B+1]
  void* out;                   // [B, rows, 512] of out_dtype
  float* out_lse;              // [B, rows] or null
  int32_t B, rows, epc, out_dtype;
  int32_t tables_ready;        // o_indptr complete before the partial kernel started: read before the wait
};
cudaError_t launch_merge_entries(const EntryMergeParams& p, cudaStream_t stream);

struct MergeParams {
  const float* partials;
  const float* lse;
  const int32_t* o_indptr;
  void* out;
  float* out_lse;
  int32_t B, rows;  // rows = q_len * H
  int32_t out_dtype;
};

// The cache write of a layer call: token i of request b's q_len new tokens goes to logical
// position context_lens[b] - q_len + i.
struct AppendParams {
  const uint16_t* ckv_new;     // [B, q_len, 512]
  const uint16_t* kpe_new;     // [B, q_len, 64]
  const int32_t* block_table;  // [B, max_blocks]
  const int32_t* context_lens; // [B]
  uint16_t* ckv;               // [num_blocks, bs, 512]
  uint16_t* kpe;               // [num_blocks, bs, 64]
  int32_t B, q_len, bs, max_blocks, num_blocks;
};

// Merge of each request's partials, then the unembed W_UV^T of each head.
struct UnembedParams {
  const float* partials;       // [N, q_len, H, 512] normalized O, or [E, q_len, H, 512] pair entries' O
  const float* lse;            // [N, q_len, H] log2 LSE, or [E, 2, q_len, H, 2] entries' (m, l)
  const int32_t* o_indptr;     // [B+1]
  const uint16_t* w_uv_t;      // [H, 512, v_head]
  void* out;                   // [B, q_len, H, v_head] of out_dtype
  float* out_lse;              // [B, q_len, H] or null
  int32_t B, q_len, H, v_head, out_dtype;
  int32_t entries;             // 1: pair entries (epc per chunk), 0: chunk partials (epc 1)
  int32_t epc;
  int32_t tables_ready;        // o_indptr complete before the preceding kernel started: read before the wait
};

// Launchers return cudaSuccess or the launch error. grid.x = cluster of
// `cluster` CTAs, grid.y = chunks, grid.z = row groups.
cudaError_t launch_partial_simt(const CUtensorMap& tm_ckv, const CUtensorMap& tm_kpe, const PartialParams& p,
                                int num_chunks, int cluster, bool bf16, cudaStream_t stream);
// tm_pages: 4D map of the ckv cache whose box is one half (256 columns) of a page;
// tm_kpe_half: kpe boxes of 32 columns with the 64-byte swizzle.
cudaError_t launch_partial_tc(const CUtensorMap& tm_ckv, const CUtensorMap& tm_kpe, const CUtensorMap& tm_pages,
                              const CUtensorMap& tm_kpe_half, const PartialParams& p, int num_chunks, int cluster,
                              bool bf16, cudaStream_t stream);
cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream);
// 128-token-tile tensor-core kernel for CTAs of at most 16 rows (fp16, bf16, or E4M3 caches),
// CTAs in pairs that split the latent columns (cluster of 2..16 CTAs).
// tm_kpe_half: kpe boxes of 32 columns with the 64-byte swizzle.
bool tc128_supports(int total_rows, bool bf16, int cluster);
cudaError_t launch_partial_tc128(const CUtensorMap& tm_pages, const CUtensorMap& tm_kpe_half, const PartialParams& p,
                                 int num_chunks, int cluster, bool bf16, cudaStream_t stream);
int tc128_max_active_clusters(int cluster);
// 64-token-tile tensor-core kernel for groups of 128 rows (q_len * H > 16, the last group
// padded), fp16 or bf16, each group on a cluster of one CTA pair that split the latent columns.
bool mh_supports(int total_rows, int cluster);
// The 128-row groups without a score exchange (xchg16 == 2): every CTA of a pair computes the full scores.
cudaError_t launch_partial_mh_nx(const CUtensorMap& tm_pages, const CUtensorMap& tm_kpe_half, const PartialParams& p,
                                 int num_chunks, bool bf16, cudaStream_t stream);
cudaError_t mh_nx_read_clear_error(uint32_t* out);
cudaError_t launch_partial_mh(const CUtensorMap& tm_pages, const CUtensorMap& tm_kpe_half, const PartialParams& p,
                              int num_chunks, bool bf16, cudaStream_t stream);

// Query rows per CTA for q_len x H rows (SIMT: always 16).
int simt_rows_per_cta();
int tc_rows_per_cta(int total_rows, bool bf16);
// Occupancy: co-resident clusters of `cluster` CTAs of the tensor-core kernel.
int tc_max_active_clusters(int cluster, int rows_per_cta, bool bf16);

cudaError_t simt_read_clear_error(uint32_t* out);
cudaError_t tc_read_clear_error(uint32_t* out);
cudaError_t tc128_read_clear_error(uint32_t* out);
cudaError_t mh_read_clear_error(uint32_t* out);
cudaError_t wrap_read_clear_error(uint32_t* out);

cudaError_t launch_cache_append(const AppendParams& p, cudaStream_t stream);
cudaError_t launch_merge_unembed(const UnembedParams& p, bool w_bf16, cudaStream_t stream);

}  // namespace mla
