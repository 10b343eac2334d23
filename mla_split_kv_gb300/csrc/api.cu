// C ABI entry points: argument checks (before any launch), TMA tensor-map
// setup, kernel dispatch, launch counters and the device error word.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "mla_split_kv.h"

namespace {

std::atomic<uint64_t> g_counters[MLA_NUM_COUNTERS];
std::atomic<uint64_t> g_timeout_ns{2000000000ull};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, fetched through the runtime so that the
// library itself does not link the driver library.
EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2D map over a [rows, cols] 16-bit matrix, boxes of 64 columns x box_rows
// rows, 128-byte swizzle (the layout both partial kernels read).
struct MapKey {
  const void* base;
  uint64_t rows, cols;
  uint32_t box_rows;
  int dtype;
  int device;
  int kind;  // 0: the 2D map; 1: the page map of the ckv cache (see page_map); 2: the kpe half map;
             // 3 / 4: the ckv / kpe half maps of an E4M3 cache (bytes, no swizzle)
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  bool valid;
};
std::mutex g_map_mu;
MapEntry g_maps[64];
int g_map_next = 0;

bool same(const MapKey& a, const MapKey& b) {
  return a.base == b.base && a.rows == b.rows && a.cols == b.cols && a.box_rows == b.box_rows && a.dtype == b.dtype &&
         a.device == b.device && a.kind == b.kind;
}

bool encode_map(CUtensorMap* out, const MapKey& key);

bool tensor_map(CUtensorMap* out, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows, int dtype) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  return encode_map(out, MapKey{base, rows, cols, box_rows, dtype, dev, 0});
}

// 4D map over the [rows, 512] ckv cache seen as (64 columns, 8 rows, 8 column
// blocks, rows / 8 row groups), boxes of (64, 8, 4, box_rows / 8): one box is
// the 256 columns of one half of a page, landing as row groups of four
// swizzled [8 x 64] atoms (the layout the paired tensor-core kernel reads).
bool page_map(CUtensorMap* out, const void* base, uint64_t rows, uint32_t box_rows, int dtype) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  return encode_map(out, MapKey{base, rows, static_cast<uint64_t>(mla::kRank), box_rows, dtype, dev, 1});
}
// 2D map over the [rows, 64] kpe cache with boxes of 32 columns x box_rows rows
// and the 64-byte swizzle: one half of the rope columns of a page, rows of 64
// bytes (two K=16 steps of a K-major tensor-core operand).
// The maps of an E4M3 cache: a CTA's half of each row (ckv 256 of 512 columns, kpe 32 of 64), bytes.
bool fp8_half_map(CUtensorMap* out, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows, int kind) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  return encode_map(out, MapKey{base, rows, cols, box_rows, MLA_E4M3, dev, kind});
}

bool kpe_half_map(CUtensorMap* out, const void* base, uint64_t rows, uint32_t box_rows, int dtype) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  return encode_map(out, MapKey{base, rows, static_cast<uint64_t>(mla::kRope), box_rows, dtype, dev, 2});
}

bool encode_map(CUtensorMap* out, const MapKey& key) {
  std::lock_guard<std::mutex> lock(g_map_mu);
  for (auto& e : g_maps)
    if (e.valid && same(e.key, key)) {
      *out = e.map;
      return true;
    }
  EncodeTiledFn enc = encoder();
  if (enc == nullptr) return false;
  CUtensorMap m;
  std::memset(&m, 0, sizeof(m));
  const CUtensorMapDataType dt =
      key.dtype == MLA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r;
  if (key.kind == 3 || key.kind == 4) {
    // E4M3 bytes: [rows][cols] with one byte an element; a box is one CTA's half of the row's columns
    // (256 of the 512 latent, 32 of the 64 rope) for box_rows rows, landing unswizzled
    cuuint64_t dims[2] = {key.cols, key.rows};
    cuuint64_t strides[1] = {key.cols};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(key.cols / 2), key.box_rows};
    cuuint32_t estr[2] = {1, 1};
    r = enc(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(key.base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else if (key.kind == 0) {
    cuuint64_t dims[2] = {key.cols, key.rows};
    cuuint64_t strides[1] = {key.cols * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(mla::kBoxCols), key.box_rows};
    cuuint32_t estr[2] = {1, 1};
    r = enc(&m, dt, 2, const_cast<void*>(key.base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else if (key.kind == 2) {
    cuuint64_t dims[2] = {key.cols, key.rows};
    cuuint64_t strides[1] = {key.cols * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(mla::kRope / 2), key.box_rows};
    cuuint32_t estr[2] = {1, 1};
    r = enc(&m, dt, 2, const_cast<void*>(key.base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    if (key.rows % 8 != 0 || key.box_rows % 8 != 0) return false;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(mla::kBoxCols), 8, key.cols / mla::kBoxCols, key.rows / 8};
    cuuint64_t strides[3] = {key.cols * 2, mla::kBoxCols * 2, key.cols * 2 * 8};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(mla::kBoxCols), 8, 4u, key.box_rows / 8};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    r = enc(&m, dt, 4, const_cast<void*>(key.base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) return false;
  g_maps[g_map_next] = MapEntry{key, m, true};
  g_map_next = (g_map_next + 1) % 64;
  *out = m;
  return true;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

mla_status_t reject(mla_status_t s) {
  g_counters[MLA_CTR_REJECTED].fetch_add(1, std::memory_order_relaxed);
  return s;
}

bool valid_heads(int32_t H) { return H == 16 || H == 64 || H == 128; }

// Cluster size when the caller leaves it to the library: enough CTAs to cover
// the SMs once, at most 16.
int default_cluster(int64_t grid_yz) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  int C = 1;
  while (C < 16 && static_cast<int64_t>(C) * 2 * grid_yz <= sms) C *= 2;
  return C;
}

}  // namespace

extern "C" {

mla_status_t mla_device_query(int32_t device, mla_device_info_t* info) {
  if (info == nullptr) return MLA_ERR_INVALID_ARG;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return MLA_ERR_CUDA;
  const int dev = device < 0 ? prev : device;
  if (cudaSetDevice(dev) != cudaSuccess) return MLA_ERR_CUDA;
  int sms = 0;
  mla_status_t st = MLA_OK;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) st = MLA_ERR_CUDA;
  info->num_sms = sms;
  for (int k = 0; k < 5; ++k)
    info->max_clusters[k] = (st == MLA_OK) ? mla::tc128_max_active_clusters(1 << k) : 0;
  cudaGetLastError();
  cudaSetDevice(prev);
  return st;
}

}  // extern "C"

namespace {

// Every argument check of mla_decode_partial, in one place, touching no GPU state. With
// check_workspace false the workspace fields are not looked at (mla_decode_partial_static
// supplies its own). Returns MLA_OK and the number of chunks, or the status to return.
mla_status_t check_decode(const void* q_absorbed, const void* q_pe, const void* ckv_cache, const void* kpe_cache,
                          const int32_t* block_table, const int32_t* context_lens, float scale,
                          int32_t num_partitions, const float* partials, const float* lse, const mla_decode_desc_t* d,
                          bool check_workspace, int64_t* n_chunks) {
  if (d == nullptr || q_absorbed == nullptr || q_pe == nullptr || ckv_cache == nullptr || kpe_cache == nullptr ||
      block_table == nullptr || context_lens == nullptr || partials == nullptr || lse == nullptr)
    return MLA_ERR_INVALID_ARG;
  if (d->num_requests < 1 || d->num_blocks < 1 || d->max_blocks_per_req < 1) return MLA_ERR_INVALID_ARG;
  if (!valid_heads(d->num_heads) || d->q_len < 1 || d->q_len > MLA_MAX_Q_LEN) return MLA_ERR_UNSUPPORTED;
  if (d->block_size != 16 && d->block_size != 32 && d->block_size != 64) return MLA_ERR_UNSUPPORTED;
  if (d->dtype != MLA_F16 && d->dtype != MLA_BF16 && d->dtype != MLA_E4M3) return MLA_ERR_UNSUPPORTED;
  if (d->dtype == MLA_E4M3) {
    // E4M3 caches: the two CTA-pair kernels only (16 rows: clusters of 2 or more; more rows: the 128-row
    // kernel's pairs), and a scale in [2^-24, 2^24]
    if (d->kernel == MLA_KERNEL_SIMT || d->cluster_ctas == 1) return MLA_ERR_UNSUPPORTED;
    if (d->num_heads * d->q_len > 16 && d->cluster_ctas != 0 && d->cluster_ctas != 2) return MLA_ERR_UNSUPPORTED;
    const float cs = d->cache_scale;
    if (!(cs >= 0x1p-24f && cs <= 0x1p24f)) return MLA_ERR_INVALID_ARG;  // also NaN
    if (d->score_exchange == MLA_SCORE_EXCHANGE_NONE) return MLA_ERR_UNSUPPORTED;  // 16-bit caches only
  }
  if (d->causal != 0 && d->causal != 1) return MLA_ERR_INVALID_ARG;
  if (d->tables_ready != 0 && d->tables_ready != 1) return MLA_ERR_INVALID_ARG;
  if (d->decode_merge != MLA_DECODE_MERGE_ENTRIES && d->decode_merge != MLA_DECODE_MERGE_TICKETS)
    return MLA_ERR_INVALID_ARG;
  if (d->prefix_ready != 0 && d->prefix_ready != 1) return MLA_ERR_INVALID_ARG;
  if (d->score_exchange < MLA_SCORE_EXCHANGE_EXACT || d->score_exchange > MLA_SCORE_EXCHANGE_F32)
    return MLA_ERR_INVALID_ARG;
  if (d->prefix_ready == 1 && d->tables_ready != 1) return MLA_ERR_INVALID_ARG;
  if (d->kernel < MLA_KERNEL_AUTO || d->kernel > MLA_KERNEL_TC) return MLA_ERR_INVALID_ARG;
  const int32_t C0 = d->cluster_ctas;
  if (C0 != 0 && C0 != 1 && C0 != 2 && C0 != 4 && C0 != 8 && C0 != 16) return MLA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return MLA_ERR_INVALID_ARG;
  if (d->clusters_per_chunk < 0 || d->clusters_per_chunk > 16) return MLA_ERR_INVALID_ARG;
  int64_t N;
  if (d->chunks == nullptr) {
    if (num_partitions < 1 || num_partitions > 1024) return MLA_ERR_INVALID_ARG;
    N = static_cast<int64_t>(d->num_requests) * num_partitions;
  } else {
    if (d->num_chunks < 1 || !aligned(d->chunks, 16)) return MLA_ERR_INVALID_ARG;
    N = d->num_chunks;
  }
  if (N > 65535) return MLA_ERR_UNSUPPORTED;
  if (!aligned(q_absorbed, 16) || !aligned(q_pe, 16) || !aligned(ckv_cache, 16) || !aligned(kpe_cache, 16) ||
      !aligned(partials, 16) || !aligned(lse, 4) || !aligned(block_table, 4) || !aligned(context_lens, 4))
    return MLA_ERR_INVALID_ARG;
  const uint64_t rows = static_cast<uint64_t>(d->num_blocks) * static_cast<uint64_t>(d->block_size);
  if (rows > 0x7fffffffull) return MLA_ERR_UNSUPPORTED;
  const int32_t subs = (d->clusters_per_chunk > 1) ? d->clusters_per_chunk : 1;
  if (subs > 1) {  // a partition spread over several clusters: the paired kernel with a workspace
    if (C0 == 0) return MLA_ERR_INVALID_ARG;  // the cluster size is part of that plan
    if (d->kernel == MLA_KERNEL_SIMT || !mla::tc128_supports(d->num_heads * d->q_len, d->dtype == MLA_BF16, C0))
      return MLA_ERR_UNSUPPORTED;
    if (check_workspace) {
      const uint64_t need = mla_workspace_bytes(static_cast<int32_t>(N), subs, C0, d->q_len, d->num_heads);
      if (d->workspace == nullptr || !aligned(d->workspace, 16) || d->workspace_bytes < need)
        return MLA_ERR_INVALID_ARG;
    }
    if (N * subs > 65535) return MLA_ERR_UNSUPPORTED;
  }
  *n_chunks = N;
  return MLA_OK;
}

// The fused final merge of mla_decode (all null / 0 for mla_decode_partial).
struct FusedMerge {
  const int32_t* o_indptr = nullptr;
  void* out = nullptr;
  float* out_lse = nullptr;
  int32_t out_dtype = 0;
  uint32_t* req_tickets = nullptr;
  float* lse_copy = nullptr;
};

// Cluster size the launch will use (the descriptor's, or the library's choice).
int launch_cluster(const mla_decode_desc_t* d, int64_t N) {
  const bool use_simt = (d->kernel == MLA_KERNEL_SIMT);
  const int rows_total = d->num_heads * d->q_len;
  const bool mh = !use_simt && mla::mh_supports(rows_total, d->cluster_ctas ? d->cluster_ctas : 2);
  const int nr = use_simt ? mla::simt_rows_per_cta()
                          : (mh ? 128 : mla::tc_rows_per_cta(rows_total, d->dtype == MLA_BF16));
  const int64_t groups = (rows_total + nr - 1) / nr;
  const int C = d->cluster_ctas ? d->cluster_ctas : (mh ? 2 : default_cluster(N * groups));
  return (d->dtype == MLA_E4M3 && C < 2) ? 2 : C;  // E4M3 runs on CTA pairs
}

// One launch of the partial kernel the descriptor selects (arguments already checked; N chunks;
// `spread_ws` the workspace of a spread plan), with the final merge fused when fm.out is set.
mla_status_t launch_decode(const void* q_absorbed, const void* q_pe, const void* ckv_cache, const void* kpe_cache,
                           const int32_t* block_table, const int32_t* context_lens, float scale,
                           int32_t num_partitions, float* partials, float* lse, const mla_decode_desc_t* d,
                           int64_t N, void* spread_ws, const FusedMerge& fm, bool entries_only = false) {
  const int32_t C0 = d->cluster_ctas;
  const uint64_t rows = static_cast<uint64_t>(d->num_blocks) * static_cast<uint64_t>(d->block_size);
  const bool use_simt = (d->kernel == MLA_KERNEL_SIMT);
  const bool bf16 = (d->dtype == MLA_BF16);
  const int rows_total = d->num_heads * d->q_len;
  // more than 16 rows on the tensor-core path: one CTA pair per 128 rows, the last group padded (a cluster
  // of 2 by default)
  const bool mh = !use_simt && mla::mh_supports(rows_total, C0 ? C0 : 2);
  const int nr = use_simt ? mla::simt_rows_per_cta() : (mh ? 128 : mla::tc_rows_per_cta(rows_total, bf16));
  const int64_t groups = (rows_total + nr - 1) / nr;
  const int32_t subs = (d->clusters_per_chunk > 1) ? d->clusters_per_chunk : 1;
  const int C = launch_cluster(d, N);

  CUtensorMap tm_ckv, tm_kpe, tm_pages, tm_kpe_half;
  const bool fp8 = (d->dtype == MLA_E4M3);
  if (fp8) {
    // the paired kernel takes the E4M3 half maps where it takes the 16-bit page and kpe half maps
    std::memset(&tm_ckv, 0, sizeof(tm_ckv));
    std::memset(&tm_kpe, 0, sizeof(tm_kpe));
    if (!fp8_half_map(&tm_pages, ckv_cache, rows, mla::kRank, d->block_size, 3) ||
        !fp8_half_map(&tm_kpe_half, kpe_cache, rows, mla::kRope, d->block_size, 4))
      return reject(MLA_ERR_CUDA);
  } else if (!tensor_map(&tm_ckv, ckv_cache, rows, mla::kRank, d->block_size, d->dtype) ||
             !tensor_map(&tm_kpe, kpe_cache, rows, mla::kRope, d->block_size, d->dtype) ||
             !page_map(&tm_pages, ckv_cache, rows, d->block_size, d->dtype) ||
             !kpe_half_map(&tm_kpe_half, kpe_cache, rows, d->block_size, d->dtype)) {
    return reject(MLA_ERR_CUDA);
  }
  if (fp8 && (use_simt || !(mh || mla::tc128_supports(rows_total, false, C)))) return reject(MLA_ERR_UNSUPPORTED);

  mla::PartialParams p;
  p.q_abs = static_cast<const uint16_t*>(q_absorbed);
  p.q_pe = static_cast<const uint16_t*>(q_pe);
  p.block_table = block_table;
  p.context_lens = context_lens;
  p.ckv = static_cast<const uint8_t*>(ckv_cache);
  p.kpe = static_cast<const uint8_t*>(kpe_cache);
  p.chunks = d->chunks;
  p.partials = partials;
  p.lse = lse;
  // an E4M3 cache's scale multiplies every score: folded into the score scale (one rounding; none
  // for a power of two)
  p.scale_log2 = scale * 1.4426950408889634f * (fp8 ? d->cache_scale : 1.0f);
  p.fp8 = fp8 ? 1 : 0;
  p.cache_scale = fp8 ? d->cache_scale : 1.0f;
  p.B = d->num_requests;
  p.H = d->num_heads;
  p.q_len = d->q_len;
  p.bs = d->block_size;
  p.max_blocks = d->max_blocks_per_req;
  p.num_blocks = d->num_blocks;
  p.num_parts = (d->chunks == nullptr) ? num_partitions : 1;
  p.causal = d->causal;
  p.tables_ready = d->tables_ready;
  p.prefix_ready = d->prefix_ready;
  // the 128-row kernel's pair: 0 fp32 partial scores cross, 1 fp16 ones, 2 none (each CTA computes the full
  // scores). The exact default: none on 16-bit caches with a full group of 128 rows; with fewer rows (a
  // 64-row group: half of each score product is padding) the fp32 exchange of the real rows' scores
  // measured faster, and E4M3 caches have only that way
  const bool full_group = d->num_heads * d->q_len >= 128;
  p.xchg16 = (d->score_exchange == MLA_SCORE_EXCHANGE_F16)  ? 1
             : (d->score_exchange == MLA_SCORE_EXCHANGE_F32) ? 0
             : (d->score_exchange == MLA_SCORE_EXCHANGE_NONE) ? 2
                                                              : ((d->dtype != MLA_E4M3 && full_group) ? 2 : 0);
  p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);

  p.subs = subs;
  p.ws_partials = nullptr;
  p.ws_lse = nullptr;
  p.ws_tickets = nullptr;
  p.entries_only = entries_only ? 1 : 0;
  if (subs > 1 || entries_only) {
    uint8_t* ws = static_cast<uint8_t*>(spread_ws);
    // tickets (two per chunk), then per chunk its entries, one per CTA pair (subs * cluster_ctas / 2),
    // [rows][512] fp32 each, then per entry two [rows][2] fp32 copies
    const uint64_t tickets = (static_cast<uint64_t>(N) * 2 * 4 + 255) / 256 * 256;
    const uint64_t entries = static_cast<uint64_t>(N) * subs * static_cast<uint64_t>(C / 2);
    p.ws_tickets = reinterpret_cast<uint32_t*>(ws);
    p.ws_partials = reinterpret_cast<float*>(ws + tickets);
    p.ws_lse = p.ws_partials + entries * rows_total * mla::kRank;
  }
  p.o_indptr = fm.o_indptr;
  p.out = fm.out;
  p.out_lse = fm.out_lse;
  p.out_dtype = fm.out_dtype;
  p.req_tickets = fm.req_tickets;
  p.lse_copy = fm.lse_copy;
  cudaStream_t stream = static_cast<cudaStream_t>(d->stream);
  const cudaError_t e =
      use_simt ? mla::launch_partial_simt(tm_ckv, tm_kpe, p, static_cast<int>(N), C, bf16, stream)
               : mla::launch_partial_tc(tm_ckv, tm_kpe, tm_pages, tm_kpe_half, p, static_cast<int>(N), C, bf16, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  g_counters[use_simt ? MLA_CTR_PARTIAL_SIMT : MLA_CTR_PARTIAL_TC].fetch_add(1, std::memory_order_relaxed);
  g_counters[MLA_CTR_CTAS].fetch_add(static_cast<uint64_t>(N * groups * C * subs), std::memory_order_relaxed);
  if (fm.out != nullptr) g_counters[MLA_CTR_DECODE_FUSED].fetch_add(1, std::memory_order_relaxed);
  return MLA_OK;
}

uint64_t round256(uint64_t x) { return (x + 255) / 256 * 256; }

// Workspace of the pair entries (the spread layout, also for one cluster per chunk): the chunk
// tickets, then N * k * C/2 entries of [rows][512] fp32, then their [2][rows][2] row maxima / sums.
uint64_t entries_ws_bytes(int64_t N, int32_t k, int32_t C, int32_t q_len, int32_t H) {
  if (N < 1 || C < 2 || q_len < 1 || H < 1) return 0;
  const uint64_t rows = static_cast<uint64_t>(q_len) * static_cast<uint64_t>(H);
  const uint64_t entries = static_cast<uint64_t>(N) * static_cast<uint64_t>(k > 1 ? k : 1) * (C / 2);
  return round256(static_cast<uint64_t>(N) * 2 * 4) + entries * rows * mla::kRank * 4 + entries * 2 * rows * 2 * 4;
}

}  // namespace

extern "C" {

mla_status_t mla_decode_partial(const void* q_absorbed, const void* q_pe, const void* ckv_cache,
                                const void* kpe_cache, const int32_t* block_table, const int32_t* context_lens,
                                float scale, int32_t num_partitions, float* partials, float* lse,
                                const mla_decode_desc_t* d) {
  int64_t N = 0;
  const mla_status_t chk = check_decode(q_absorbed, q_pe, ckv_cache, kpe_cache, block_table, context_lens, scale,
                                        num_partitions, partials, lse, d, true, &N);
  if (chk != MLA_OK) return reject(chk);
  return launch_decode(q_absorbed, q_pe, ckv_cache, kpe_cache, block_table, context_lens, scale, num_partitions,
                       partials, lse, d, N, d->workspace, FusedMerge{});
}

uint64_t mla_decode_workspace_bytes(int32_t num_requests, int32_t num_chunks, int32_t clusters_per_chunk,
                                    int32_t cluster_ctas, int32_t q_len, int32_t num_heads) {
  if (num_requests < 1 || num_chunks < 1 || q_len < 1 || num_heads < 1) return 0;
  const uint64_t tickets = round256(static_cast<uint64_t>(num_requests) * mla::kSliceTickets * 4);
  const uint64_t lse_copy = round256(static_cast<uint64_t>(num_chunks) * q_len * num_heads * 4);
  // one layout for both ways: the request tickets and LSE copies of the single launch, then the
  // chunk tickets and pair entries (the default path writes only the entries, never a ticket)
  return tickets + lse_copy + entries_ws_bytes(num_chunks, clusters_per_chunk, cluster_ctas, q_len, num_heads);
}

}  // extern "C"

namespace {

// The paired kernel's default way: every CTA pair writes its unnormalized part (O, row maxima and
// sums) to an entry of the workspace, laid out as mla_decode_workspace_bytes describes.
struct PairEntries {
  const float* o;   // [E, q_len, H, 512]
  const float* ml;  // [E, 2, q_len, H, 2]
  int32_t epc;      // entries per chunk
};

mla_status_t launch_pair_entries(const void* q_absorbed, const void* q_pe, const void* ckv_cache, const void* kpe_cache,
                                 const int32_t* block_table, const int32_t* context_lens, float scale,
                                 int32_t num_partitions, float* partials, float* lse, const mla_decode_desc_t* d,
                                 int64_t N, PairEntries* out) {
  const int rows_total = d->num_heads * d->q_len;
  const int32_t C = launch_cluster(d, N);
  const uint64_t head = round256(static_cast<uint64_t>(d->num_requests) * mla::kSliceTickets * 4) +
                        round256(static_cast<uint64_t>(N) * rows_total * 4);  // the TICKETS way's blocks
  const uint64_t need = head + entries_ws_bytes(N, d->clusters_per_chunk, C, d->q_len, d->num_heads);
  if (d->workspace == nullptr || !aligned(d->workspace, 16) || d->workspace_bytes < need)
    return reject(MLA_ERR_INVALID_ARG);
  uint8_t* ws = static_cast<uint8_t*>(d->workspace) + head;
  const int32_t k = d->clusters_per_chunk > 1 ? d->clusters_per_chunk : 1;
  mla_status_t st = launch_decode(q_absorbed, q_pe, ckv_cache, kpe_cache, block_table, context_lens, scale,
                                  num_partitions, partials, lse, d, N, ws, FusedMerge{}, true);
  if (st != MLA_OK) return st;
  const uint64_t entries = static_cast<uint64_t>(N) * k * (C / 2);
  out->o = reinterpret_cast<const float*>(ws + round256(static_cast<uint64_t>(N) * 2 * 4));
  out->ml = out->o + entries * rows_total * mla::kRank;
  out->epc = k * (C / 2);
  return MLA_OK;
}

}  // namespace

extern "C" {

mla_status_t mla_decode(const void* q_absorbed, const void* q_pe, const void* ckv_cache, const void* kpe_cache,
                        const int32_t* block_table, const int32_t* context_lens, float scale, int32_t num_partitions,
                        float* partials, float* lse, const int32_t* o_indptr, void* out, int32_t out_dtype,
                        float* out_lse, const mla_decode_desc_t* d) {
  int64_t N = 0;
  const mla_status_t chk = check_decode(q_absorbed, q_pe, ckv_cache, kpe_cache, block_table, context_lens, scale,
                                        num_partitions, partials, lse, d, false, &N);
  if (chk != MLA_OK) return reject(chk);
  if (o_indptr == nullptr || out == nullptr || !aligned(o_indptr, 4) || !aligned(out, 16) ||
      (out_lse != nullptr && !aligned(out_lse, 4)))
    return reject(MLA_ERR_INVALID_ARG);
  if (out_dtype != MLA_F16 && out_dtype != MLA_BF16 && out_dtype != MLA_F32) return reject(MLA_ERR_UNSUPPORTED);
  const int rows_total = d->num_heads * d->q_len;
  const bool paired = d->kernel != MLA_KERNEL_SIMT &&
                      mla::tc128_supports(rows_total, d->dtype == MLA_BF16, launch_cluster(d, N));
  const bool fused = paired && d->decode_merge == MLA_DECODE_MERGE_TICKETS;
  if (paired && !fused) {
    // the paired kernel writes every CTA pair's part to the workspace and exits; the entries merge
    // kernel, a programmatic dependent launch resident beside it, combines a request's parts
    // straight into the output
    PairEntries pe;
    mla_status_t st = launch_pair_entries(q_absorbed, q_pe, ckv_cache, kpe_cache, block_table, context_lens, scale,
                                          num_partitions, partials, lse, d, N, &pe);
    if (st != MLA_OK) return st;
    mla::EntryMergeParams mp;
    mp.ws_partials = pe.o;
    mp.ws_lse = pe.ml;
    mp.o_indptr = o_indptr;
    mp.out = out;
    mp.out_lse = out_lse;
    mp.B = d->num_requests;
    mp.rows = rows_total;
    mp.epc = pe.epc;
    mp.out_dtype = out_dtype;
    mp.tables_ready = d->tables_ready;
    if (mla::launch_merge_entries(mp, static_cast<cudaStream_t>(d->stream)) != cudaSuccess) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    g_counters[MLA_CTR_MERGE].fetch_add(1, std::memory_order_relaxed);
    return MLA_OK;
  }
  if (!fused) {
    // the partial kernel, then the merge kernel (a programmatic dependent launch), on the same stream
    if (d->clusters_per_chunk > 1) {
      const uint64_t need = mla_workspace_bytes(static_cast<int32_t>(N), d->clusters_per_chunk, d->cluster_ctas,
                                                d->q_len, d->num_heads);
      if (d->workspace == nullptr || !aligned(d->workspace, 16) || d->workspace_bytes < need)
        return reject(MLA_ERR_INVALID_ARG);
    }
    mla_status_t st = launch_decode(q_absorbed, q_pe, ckv_cache, kpe_cache, block_table, context_lens, scale,
                                    num_partitions, partials, lse, d, N, d->workspace, FusedMerge{});
    if (st != MLA_OK) return st;
    return mla_merge_states(partials, lse, o_indptr, d->num_requests, d->q_len, d->num_heads, out, out_dtype, out_lse,
                            d->stream);
  }
  const uint64_t need = mla_decode_workspace_bytes(d->num_requests, static_cast<int32_t>(N), d->clusters_per_chunk,
                                                   d->cluster_ctas, d->q_len, d->num_heads);
  if (d->workspace == nullptr || !aligned(d->workspace, 16) || d->workspace_bytes < need)
    return reject(MLA_ERR_INVALID_ARG);
  uint8_t* ws = static_cast<uint8_t*>(d->workspace);
  FusedMerge fm;
  fm.o_indptr = o_indptr;
  fm.out = out;
  fm.out_lse = out_lse;
  fm.out_dtype = out_dtype;
  fm.req_tickets = reinterpret_cast<uint32_t*>(ws);
  const uint64_t tickets = round256(static_cast<uint64_t>(d->num_requests) * mla::kSliceTickets * 4);
  fm.lse_copy = reinterpret_cast<float*>(ws + tickets);
  void* spread_ws = ws + tickets + round256(static_cast<uint64_t>(N) * rows_total * 4);
  return launch_decode(q_absorbed, q_pe, ckv_cache, kpe_cache, block_table, context_lens, scale, num_partitions,
                       partials, lse, d, N, spread_ws, fm);
}

mla_status_t mla_decode_unembed(const void* q_absorbed, const void* q_pe, const void* ckv_cache, const void* kpe_cache,
                                const int32_t* block_table, const int32_t* context_lens, float scale,
                                int32_t num_partitions, float* partials, float* lse, const int32_t* o_indptr,
                                const void* w_uv_t, int32_t w_dtype, int32_t v_head, void* out_v, int32_t out_dtype,
                                float* out_lse, const mla_decode_desc_t* d) {
  int64_t N = 0;
  const mla_status_t chk = check_decode(q_absorbed, q_pe, ckv_cache, kpe_cache, block_table, context_lens, scale,
                                        num_partitions, partials, lse, d, false, &N);
  if (chk != MLA_OK) return reject(chk);
  if (o_indptr == nullptr || out_v == nullptr || w_uv_t == nullptr || !aligned(o_indptr, 4) || !aligned(out_v, 4) ||
      !aligned(w_uv_t, 16) || (out_lse != nullptr && !aligned(out_lse, 4)))
    return reject(MLA_ERR_INVALID_ARG);
  if (v_head < 32 || v_head > 512 || v_head % 32 != 0) return reject(MLA_ERR_UNSUPPORTED);
  if (w_dtype != MLA_F16 && w_dtype != MLA_BF16) return reject(MLA_ERR_UNSUPPORTED);
  if (out_dtype != MLA_F16 && out_dtype != MLA_BF16 && out_dtype != MLA_F32) return reject(MLA_ERR_UNSUPPORTED);
  if (static_cast<int64_t>(d->num_requests) * d->q_len > 65535LL * 16) return reject(MLA_ERR_UNSUPPORTED);
  const int rows_total = d->num_heads * d->q_len;
  const bool paired = d->kernel != MLA_KERNEL_SIMT &&
                      mla::tc128_supports(rows_total, d->dtype == MLA_BF16, launch_cluster(d, N));
  if (paired && d->decode_merge == MLA_DECODE_MERGE_TICKETS) return reject(MLA_ERR_UNSUPPORTED);
  mla::UnembedParams up;
  up.o_indptr = o_indptr;
  up.w_uv_t = static_cast<const uint16_t*>(w_uv_t);
  up.out = out_v;
  up.out_lse = out_lse;
  up.B = d->num_requests;
  up.q_len = d->q_len;
  up.H = d->num_heads;
  up.v_head = v_head;
  up.out_dtype = out_dtype;
  up.tables_ready = d->tables_ready;
  if (paired) {
    // the paired kernel's pair entries, merged and unembedded by one programmatic dependent launch
    PairEntries pe;
    mla_status_t st = launch_pair_entries(q_absorbed, q_pe, ckv_cache, kpe_cache, block_table, context_lens, scale,
                                          num_partitions, partials, lse, d, N, &pe);
    if (st != MLA_OK) return st;
    up.partials = pe.o;
    up.lse = pe.ml;
    up.entries = 1;
    up.epc = pe.epc;
  } else {
    // chunk partials, then their merge with the unembed
    if (d->clusters_per_chunk > 1) {
      const uint64_t need = mla_workspace_bytes(static_cast<int32_t>(N), d->clusters_per_chunk, d->cluster_ctas,
                                                d->q_len, d->num_heads);
      if (d->workspace == nullptr || !aligned(d->workspace, 16) || d->workspace_bytes < need)
        return reject(MLA_ERR_INVALID_ARG);
    }
    mla_status_t st = launch_decode(q_absorbed, q_pe, ckv_cache, kpe_cache, block_table, context_lens, scale,
                                    num_partitions, partials, lse, d, N, d->workspace, FusedMerge{});
    if (st != MLA_OK) return st;
    up.partials = partials;
    up.lse = lse;
    up.entries = 0;
    up.epc = 1;
  }
  if (mla::launch_merge_unembed(up, w_dtype == MLA_BF16, static_cast<cudaStream_t>(d->stream)) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  g_counters[MLA_CTR_WRAP].fetch_add(1, std::memory_order_relaxed);
  return MLA_OK;
}

}  // extern "C"

namespace {

// Scratch of mla_decode_partial_static: one statically sized array per device
// (the module is loaded on each device that uses it). Its address is looked up
// once per device and process; it is cleared then, since the chunk tickets
// must start at zero (every call that completes leaves them at zero again),
// and again by mla_check_device_errors when it finds the error word set (an
// aborted call may leave tickets counted).
static __device__ __align__(256) uint8_t g_static_workspace[MLA_STATIC_WORKSPACE_BYTES];
constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_addr[kMaxDevices] = {};

mla_status_t static_workspace(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static_addr[dev] == nullptr) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_static_workspace) != cudaSuccess || addr == nullptr) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    if (cudaMemset(addr, 0, MLA_STATIC_WORKSPACE_BYTES) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    g_static_addr[dev] = addr;
  }
  *out = g_static_addr[dev];
  return MLA_OK;
}

// Zero the current device's static scratch if it has been set up (after a
// device error, when a call may have stopped with tickets counted).
bool clear_static_workspace() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static_addr[dev] == nullptr) return true;
  return cudaMemset(g_static_addr[dev], 0, MLA_STATIC_WORKSPACE_BYTES) == cudaSuccess &&
         cudaDeviceSynchronize() == cudaSuccess;
}

}  // namespace

extern "C" {

mla_status_t mla_decode_partial_static(const void* q_absorbed, const void* q_pe, const void* ckv_cache,
                                       const void* kpe_cache, const int32_t* block_table,
                                       const int32_t* context_lens, float scale, int32_t num_partitions,
                                       float* partials, float* lse, const mla_decode_desc_t* d) {
  int64_t N = 0;
  const mla_status_t chk = check_decode(q_absorbed, q_pe, ckv_cache, kpe_cache, block_table, context_lens, scale,
                                        num_partitions, partials, lse, d, false, &N);
  if (chk != MLA_OK) return reject(chk);
  mla_decode_desc_t dd = *d;
  dd.workspace = nullptr;
  dd.workspace_bytes = 0;
  if (dd.clusters_per_chunk > 1) {  // a valid spread plan: the library's scratch stands in for the workspace
    const uint64_t need =
        mla_workspace_bytes(static_cast<int32_t>(N), dd.clusters_per_chunk, dd.cluster_ctas, dd.q_len, dd.num_heads);
    if (need > MLA_STATIC_WORKSPACE_BYTES) return reject(MLA_ERR_CAPACITY);
    void* ws = nullptr;
    const mla_status_t st = static_workspace(&ws);
    if (st != MLA_OK) return st;
    dd.workspace = ws;
    dd.workspace_bytes = MLA_STATIC_WORKSPACE_BYTES;
  }
  return mla_decode_partial(q_absorbed, q_pe, ckv_cache, kpe_cache, block_table, context_lens, scale, num_partitions,
                            partials, lse, &dd);
}

uint64_t mla_workspace_bytes(int32_t num_chunks, int32_t clusters_per_chunk, int32_t cluster_ctas, int32_t q_len,
                             int32_t num_heads) {
  if (clusters_per_chunk <= 1 || num_chunks < 1 || cluster_ctas < 2 || q_len < 1 || num_heads < 1) return 0;
  const uint64_t n = static_cast<uint64_t>(num_chunks), k = static_cast<uint64_t>(clusters_per_chunk);
  const uint64_t rows = static_cast<uint64_t>(q_len) * static_cast<uint64_t>(num_heads);
  const uint64_t entries = n * k * static_cast<uint64_t>(cluster_ctas / 2);
  const uint64_t tickets = (n * 2 * 4 + 255) / 256 * 256;
  return tickets + entries * rows * mla::kRank * 4 + entries * 2 * rows * 2 * 4;
}

mla_status_t mla_merge_states(const float* partials, const float* lse, const int32_t* o_indptr, int32_t B,
                              int32_t q_len, int32_t num_heads, void* out, int32_t out_dtype, float* out_lse,
                              void* stream) {
  if (partials == nullptr || lse == nullptr || o_indptr == nullptr || out == nullptr) return reject(MLA_ERR_INVALID_ARG);
  if (B < 1 || B > (1 << 24)) return reject(MLA_ERR_INVALID_ARG);
  if (!valid_heads(num_heads) || q_len < 1 || q_len > MLA_MAX_Q_LEN) return reject(MLA_ERR_UNSUPPORTED);
  if (out_dtype != MLA_F16 && out_dtype != MLA_BF16 && out_dtype != MLA_F32) return reject(MLA_ERR_UNSUPPORTED);
  if (!aligned(partials, 16) || !aligned(lse, 4) || !aligned(o_indptr, 4) || !aligned(out, 16) ||
      (out_lse != nullptr && !aligned(out_lse, 4)))
    return reject(MLA_ERR_INVALID_ARG);
  mla::MergeParams p;
  p.partials = partials;
  p.lse = lse;
  p.o_indptr = o_indptr;
  p.out = out;
  p.out_lse = out_lse;
  p.B = B;
  p.rows = q_len * num_heads;
  p.out_dtype = out_dtype;
  const cudaError_t e = mla::launch_merge(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  g_counters[MLA_CTR_MERGE].fetch_add(1, std::memory_order_relaxed);
  return MLA_OK;
}

mla_status_t mla_cache_append(const void* ckv_new, const void* kpe_new, const int32_t* block_table,
                              const int32_t* context_lens, int32_t B, int32_t q_len, int32_t block_size,
                              int32_t num_blocks, int32_t max_blocks_per_req, void* ckv_cache, void* kpe_cache,
                              void* stream) {
  if (ckv_new == nullptr || kpe_new == nullptr || block_table == nullptr || context_lens == nullptr ||
      ckv_cache == nullptr || kpe_cache == nullptr)
    return reject(MLA_ERR_INVALID_ARG);
  if (B < 1 || B > (1 << 24) || num_blocks < 1 || max_blocks_per_req < 1) return reject(MLA_ERR_INVALID_ARG);
  if (q_len < 1 || q_len > MLA_MAX_Q_LEN) return reject(MLA_ERR_UNSUPPORTED);
  if (block_size != 16 && block_size != 32 && block_size != 64) return reject(MLA_ERR_UNSUPPORTED);
  if (!aligned(ckv_new, 16) || !aligned(kpe_new, 16) || !aligned(ckv_cache, 16) || !aligned(kpe_cache, 16) ||
      !aligned(block_table, 4) || !aligned(context_lens, 4))
    return reject(MLA_ERR_INVALID_ARG);
  mla::AppendParams p;
  p.ckv_new = static_cast<const uint16_t*>(ckv_new);
  p.kpe_new = static_cast<const uint16_t*>(kpe_new);
  p.block_table = block_table;
  p.context_lens = context_lens;
  p.ckv = static_cast<uint16_t*>(ckv_cache);
  p.kpe = static_cast<uint16_t*>(kpe_cache);
  p.B = B;
  p.q_len = q_len;
  p.bs = block_size;
  p.max_blocks = max_blocks_per_req;
  p.num_blocks = num_blocks;
  if (mla::launch_cache_append(p, static_cast<cudaStream_t>(stream)) != cudaSuccess) return MLA_ERR_CUDA;
  g_counters[MLA_CTR_WRAP].fetch_add(1, std::memory_order_relaxed);
  return MLA_OK;
}

mla_status_t mla_merge_unembed(const float* partials, const float* lse, const int32_t* o_indptr, int32_t B,
                               int32_t q_len, int32_t num_heads, const void* w_uv_t, int32_t w_dtype, int32_t v_head,
                               void* out, int32_t out_dtype, float* out_lse, void* stream) {
  if (partials == nullptr || lse == nullptr || o_indptr == nullptr || w_uv_t == nullptr || out == nullptr)
    return reject(MLA_ERR_INVALID_ARG);
  if (B < 1 || B > (1 << 24)) return reject(MLA_ERR_INVALID_ARG);
  if (!valid_heads(num_heads) || q_len < 1 || q_len > MLA_MAX_Q_LEN) return reject(MLA_ERR_UNSUPPORTED);
  if (v_head < 32 || v_head > 512 || v_head % 32 != 0) return reject(MLA_ERR_UNSUPPORTED);
  if (w_dtype != MLA_F16 && w_dtype != MLA_BF16) return reject(MLA_ERR_UNSUPPORTED);
  if (out_dtype != MLA_F16 && out_dtype != MLA_BF16 && out_dtype != MLA_F32) return reject(MLA_ERR_UNSUPPORTED);
  if (static_cast<int64_t>(B) * q_len > 65535LL * 16) return reject(MLA_ERR_UNSUPPORTED);
  if (!aligned(partials, 16) || !aligned(lse, 4) || !aligned(o_indptr, 4) || !aligned(w_uv_t, 16) ||
      !aligned(out, 4) || (out_lse != nullptr && !aligned(out_lse, 4)))
    return reject(MLA_ERR_INVALID_ARG);
  mla::UnembedParams p;
  p.partials = partials;
  p.lse = lse;
  p.o_indptr = o_indptr;
  p.w_uv_t = static_cast<const uint16_t*>(w_uv_t);
  p.out = out;
  p.out_lse = out_lse;
  p.B = B;
  p.q_len = q_len;
  p.H = num_heads;
  p.v_head = v_head;
  p.out_dtype = out_dtype;
  p.entries = 0;
  p.epc = 1;
  p.tables_ready = 0;
  if (mla::launch_merge_unembed(p, w_dtype == MLA_BF16, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  g_counters[MLA_CTR_WRAP].fetch_add(1, std::memory_order_relaxed);
  return MLA_OK;
}

mla_status_t mla_check_device_errors(void* stream, uint32_t* code_out) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MLA_ERR_CUDA;
  uint32_t a = 0, b = 0, c = 0, e = 0, f = 0, g = 0;
  if (mla::simt_read_clear_error(&a) != cudaSuccess || mla::tc_read_clear_error(&b) != cudaSuccess ||
      mla::tc128_read_clear_error(&c) != cudaSuccess || mla::mh_read_clear_error(&e) != cudaSuccess ||
      mla::wrap_read_clear_error(&f) != cudaSuccess || mla::mh_nx_read_clear_error(&g) != cudaSuccess)
    return MLA_ERR_CUDA;
  const uint32_t code = a | b | c | e | f | g;
  if (code_out != nullptr) *code_out = code;
  if (code != 0 && !clear_static_workspace()) return MLA_ERR_CUDA;
  if (code & mla::MLA_DEVERR_TIMEOUT) return MLA_ERR_TIMEOUT;
  if (code != 0) return MLA_ERR_DEVICE_CHECK;
  return MLA_OK;
}

void mla_get_counters(uint64_t* out, int32_t n) {
  if (out == nullptr) return;
  for (int32_t i = 0; i < n && i < MLA_NUM_COUNTERS; ++i) out[i] = g_counters[i].load(std::memory_order_relaxed);
}

void mla_reset_counters(void) {
  for (auto& c : g_counters) c.store(0, std::memory_order_relaxed);
}

void mla_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns, std::memory_order_relaxed); }

size_t mla_partials_bytes(int32_t num_slots, int32_t q_len, int32_t num_heads) {
  if (num_slots < 0 || q_len < 0 || num_heads < 0) return 0;
  return static_cast<size_t>(num_slots) * q_len * num_heads * mla::kRank * sizeof(float);
}

size_t mla_lse_bytes(int32_t num_slots, int32_t q_len, int32_t num_heads) {
  if (num_slots < 0 || q_len < 0 || num_heads < 0) return 0;
  return static_cast<size_t>(num_slots) * q_len * num_heads * sizeof(float);
}

const char* mla_status_string(mla_status_t s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_TIMEOUT: return "device wait timed out";
    case MLA_ERR_DEVICE_CHECK: return "device data check failed";
    case MLA_ERR_CAPACITY: return "plan capacity too small";
  }
  return "unknown status";
}

int32_t mla_version(void) { return 1; }

}  // extern "C"
