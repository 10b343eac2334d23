// The steps either side of attention in a decode layer call, sm_103a.
//
// "[kernel] Wire MLA split-KV decode" (vllm-metal PR #601), *Bench*: the MLA
// wrapper writes the new token's latent into the paged cache before attention
// and unembeds the attention output after it. "feat(core): matrix-absorbed MLA
// decode over a compressed-latent KV cache" (mlxcel PR #995), *What changed*:
// the output side of the fold is W_UV^T [H, r, v_head], applied to the latent
// attention output of each head.
//
//  - mla_cache_append_kernel: one warp per new token copies its 512 latent and
//    64 rope values (1152 bytes, 16-byte pieces) to the token's physical cache
//    row. A pure copy: HBM-bound, 2 x 1152 bytes per token.
//  - mla_merge_unembed_kernel: per (head, 32 value columns, 16 rows of that
//    head) one CTA merges the rows' partials over all 512 latent columns in the
//    merge kernel's arithmetic (so the fp32 latent is the bits
//    mla_merge_states would give, never rounded): each warp takes the LSE
//    maximum, the weights and their sum of two rows, the weights go to shared
//    memory in pieces of 128 partials, and each thread sums its two latent
//    columns over the partials in order with 32 loads in flight (the first
//    round issued before the maxima are known). The head's W_UV^T slice
//    [512 x 32] is staged while the preceding kernel finishes, each warp
//    keeping its 64 rows of it in registers; the product runs in fp32 in a
//    fixed order (eight chunks of 64 d, each in order, one per warp, then the
//    chunk sums in order) over the real rows only, rounded once to the output
//    type. A single-token decode call is latency-bound here: a few dependent
//    L2 round trips, not bytes.
#include "device_common.cuh"

namespace mla {

namespace {

constexpr int kAppendWarps = 4;

__global__ void __launch_bounds__(kAppendWarps * 32) mla_cache_append_kernel(const AppendParams p) {
  // the kernel after it (the layer call's decode) may start at once: it reads nothing this kernel writes
  // before waiting for it to complete. This kernel waits for the one before it (which may produce the new
  // tokens) before reading anything.
  pdl_launch_dependents();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long tok = static_cast<long long>(blockIdx.x) * kAppendWarps + warp;  // b * q_len + i
  if (tok >= static_cast<long long>(p.B) * p.q_len) return;
  const int b = static_cast<int>(tok / p.q_len), i = static_cast<int>(tok % p.q_len);
  const int t = p.context_lens[b] - p.q_len + i;  // the window's rows are the last q_len positions
  if (t < 0) return;
  const int pg = t / p.bs;
  const int pid = (pg < p.max_blocks) ? p.block_table[static_cast<long long>(b) * p.max_blocks + pg] : -1;
  if (pid < 0 || pid >= p.num_blocks) {  // outside the table or the pool: nothing is written
    if (lane == 0) flag_error(MLA_DEVERR_BAD_PAGE);
    return;
  }
  const long long row = static_cast<long long>(pid) * p.bs + t % p.bs;
  const uint4* src_c = reinterpret_cast<const uint4*>(p.ckv_new + tok * kRank);
  uint4* dst_c = reinterpret_cast<uint4*>(p.ckv + row * kRank);
#pragma unroll
  for (int x = lane; x < kRank * 2 / 16; x += 32) dst_c[x] = src_c[x];
  if (lane < kRope * 2 / 16)
    reinterpret_cast<uint4*>(p.kpe + row * kRope)[lane] = reinterpret_cast<const uint4*>(p.kpe_new + tok * kRope)[lane];
}

constexpr int kUnThreads = 256;
constexpr int kUnRows = 16;  // rows of one head per CTA
constexpr int kUnCols = 32;  // value columns per CTA
constexpr int kUnChunks = kUnThreads / 32;  // the d range in 8 chunks of 64, one per warp
constexpr int kUnDper = kRank / kUnChunks;  // d values per chunk
constexpr uint32_t kUnPartOff = kUnRows * kRank * 4 + kRank * kUnCols * 2;  // after the latent rows + W slice
constexpr int kUnPiece = 128;  // partial weights held in shared memory at a time, per row
constexpr int kUnDepth = 32;   // partial values a thread has in flight
constexpr uint32_t kUnWgtOff = kUnPartOff + kUnChunks * kUnRows * kUnCols * 4;  // after the chunk sums
constexpr uint32_t kUnRowOff = kUnWgtOff + 2 * kUnRows * kUnPiece * 4;  // after the weights and sums l
constexpr uint32_t kUnSmem = kUnRowOff + 5 * kUnRows * 4;  // + each row's range, slot row, sum, maximum: 96.3 KB
static_assert(kRank / 2 == kUnThreads, "one thread per pair of latent columns");
static_assert(kUnPiece % 32 == 0, "whole warps of weights");
static_assert(kRank * 4 % kUnThreads == 0, "whole 16-byte pieces of the W slice per thread");

// Two sources of a row's parts: chunk partials (normalized O with its log2 LSE; the merge is
// mla_merge_states' arithmetic, one chain per column in partial order) or the paired kernel's pair
// entries (unnormalized O with the pair's row maximum m and sum l relative to m; the merge is the
// entries merge's arithmetic: eight groups of entries, entry e in group (e - first) mod 8, each group
// summed in order, then the groups added as ((0+1)+(2+3))+((4+5)+(6+7))). Either way the fp32
// latent is the bits the stand-alone merge writes.
template <bool BF16, bool kEntries>
__global__ void __launch_bounds__(kUnThreads, 1) mla_merge_unembed_kernel(const UnembedParams p) {
  extern __shared__ uint8_t smem_raw[];
  float* lat = reinterpret_cast<float*>(smem_raw);                          // [16][512] fp32
  uint16_t* wsl = reinterpret_cast<uint16_t*>(smem_raw + kUnRows * kRank * 4);  // [512][32] 16-bit
  int* row_lo = reinterpret_cast<int*>(smem_raw + kUnRowOff);
  int* row_n = row_lo + kUnRows;
  int* row_r = row_n + kUnRows;
  float* row_den = reinterpret_cast<float*>(row_r + kUnRows);
  float* row_m = row_den + kUnRows;
  float* wgt = reinterpret_cast<float*>(smem_raw + kUnWgtOff);  // [16 rows][kUnPiece] weights
  float* lsum = wgt + kUnRows * kUnPiece;                        // [16 rows][kUnPiece] entries' sums l
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int h = blockIdx.x, vblk = blockIdx.y;
  const int rows_total = p.q_len * p.H;
  const int R = p.B * p.q_len;  // rows of head h
  const int rr0 = blockIdx.z * kUnRows;
  const int nrows = min(kUnRows, R - rr0);
  // each row's parts: slots lo .. lo + n - 1 (row rr of head h = query row i of request b)
  auto row_ranges = [&]() {
    if (tid < nrows) {
      const int rr = rr0 + tid, b = rr / p.q_len, i = rr % p.q_len;
      const int lo = __ldg(p.o_indptr + b) * p.epc;
      row_lo[tid] = lo;
      row_n[tid] = __ldg(p.o_indptr + b + 1) * p.epc - lo;
      row_r[tid] = i * p.H + h;
    }
  };
  if (p.tables_ready) row_ranges();  // the offsets were complete before the preceding kernel started
  // this head's W_UV^T columns [32 vblk, 32 vblk + 32): 512 rows of 64 bytes. The weights are no output
  // of the preceding kernel: they are staged while it finishes, all of a thread's loads in flight at once
  const uint16_t* wsrc = p.w_uv_t + (static_cast<long long>(h) * kRank) * p.v_head + vblk * kUnCols;
  {
    constexpr int kPer = kRank * 4 / kUnThreads;  // 16-byte pieces per thread: 8
    uint4 wv[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int x = tid + u * kUnThreads, d = x >> 2, q = x & 3;
      wv[u] = *reinterpret_cast<const uint4*>(wsrc + static_cast<long long>(d) * p.v_head + q * 8);
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int x = tid + u * kUnThreads, d = x >> 2, q = x & 3;
      reinterpret_cast<uint4*>(wsl + d * kUnCols)[q] = wv[u];
    }
  }
  __syncthreads();
  float wreg[kUnDper];  // W[64 w + dd][32 vblk + lane]
#pragma unroll
  for (int dd = 0; dd < kUnDper; ++dd) wreg[dd] = h2f<BF16>(wsl[(w * kUnDper + dd) * kUnCols + lane]);
  pdl_wait();  // a programmatic dependent of the partial kernel: its parts are complete after this
  pdl_launch_dependents();
  if (!p.tables_ready) row_ranges();
  __syncthreads();
  // the merged latent: thread tid owns latent columns 2 tid, 2 tid + 1 of every row; warp w takes rows
  // w, w + 8 for the maxima, the weights and their sum
  const long long stride = static_cast<long long>(rows_total) * kRank;  // one slot's values
  // a part's (LSE, 0) or (m, l)
  auto part_ml = [&](int k, int j) -> float2 {
    if (kEntries)
      return __ldcg(reinterpret_cast<const float2*>(p.lse + static_cast<long long>(row_lo[k] + j) * 4 * rows_total +
                                                    row_r[k] * 2));
    return make_float2(__ldcg(p.lse + static_cast<long long>(row_lo[k] + j) * rows_total + row_r[k]), 0.f);
  };
  float2 v[kUnDepth];
  // values of parts k, j0 .. j0 + kUnDepth - 1 for this thread's columns, all loads in flight at once
  auto load_values = [&](int k, int j0) {
    const float* src = p.partials + static_cast<long long>(row_lo[k]) * stride +
                       static_cast<long long>(row_r[k]) * kRank + 2 * tid;
#pragma unroll
    for (int jj = 0; jj < kUnDepth; ++jj)
      v[jj] = (j0 + jj < row_n[k]) ? __ldcg(reinterpret_cast<const float2*>(src + (j0 + jj) * stride))
                                   : make_float2(0.f, 0.f);
  };
  if (nrows > 0) load_values(0, 0);  // the first round goes out before the maxima are known
  // the weights (and the entries' sums) of parts j0 .. j0 + kUnPiece - 1 of row k, by one warp
  auto put_weights = [&](int k, int j0, float m, const float2* ml) {
#pragma unroll
    for (int t = 0; t < kUnPiece / 32; ++t) {
      const int jj = lane + 32 * t;
      const float2 x = (ml != nullptr) ? ml[t] : ((j0 + jj < row_n[k]) ? part_ml(k, j0 + jj) : make_float2(-INFINITY, 0.f));
      wgt[k * kUnPiece + jj] = (x.x == -INFINITY) ? 0.f : exp2f(x.x - m);
      if (kEntries) lsum[k * kUnPiece + jj] = (j0 + jj < row_n[k]) ? x.y : 0.f;
    }
  };
  // the weight sum over parts j0 .. j0 + cnt - 1 of row k, continuing `den` (eight group sums for entries)
  auto add_den = [&](int k, int cnt, float* den) {
    for (int j0 = 0; j0 < cnt; j0 += 8) {
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        if (j0 + g < cnt) {
          if (kEntries)
            den[g] = fmaf(wgt[k * kUnPiece + j0 + g], lsum[k * kUnPiece + j0 + g], den[g]);
          else
            den[0] += wgt[k * kUnPiece + j0 + g];
        }
      }
    }
  };
  {
    float2 ml[2][kUnPiece / 32];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int k = w + 8 * s;
#pragma unroll
      for (int t = 0; t < kUnPiece / 32; ++t) {
        const int j = lane + 32 * t;
        ml[s][t] = (k < nrows && j < row_n[k]) ? part_ml(k, j) : make_float2(-INFINITY, 0.f);
      }
    }
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int k = w + 8 * s;
      if (k >= nrows) continue;
      float m = -INFINITY;
#pragma unroll
      for (int t = 0; t < kUnPiece / 32; ++t) m = fmaxf(m, ml[s][t].x);
      for (int j = kUnPiece + lane; j < row_n[k]; j += 32) m = fmaxf(m, part_ml(k, j).x);  // more than a piece
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      put_weights(k, 0, m, ml[s]);
      if (lane == 0) row_m[k] = m;
    }
  }
  __syncthreads();
  float2* lat2 = reinterpret_cast<float2*>(lat);
  for (int k = 0; k < nrows; ++k) {
    const int n = row_n[k];
    float2 acc[kEntries ? 8 : 1];
#pragma unroll
    for (int g = 0; g < (kEntries ? 8 : 1); ++g) acc[g] = make_float2(0.f, 0.f);
    float den[kEntries ? 8 : 1];
#pragma unroll
    for (int g = 0; g < (kEntries ? 8 : 1); ++g) den[g] = 0.f;
    for (int j0 = 0; j0 < n; j0 += kUnPiece) {
      if (j0 > 0) {  // a row with more parts than a piece: its next weights, by warp 0
        __syncthreads();  // the row's previous weights are read
        if (w == 0) put_weights(k, j0, row_m[k], nullptr);
        __syncthreads();
      }
      const int cnt = min(kUnPiece, n - j0);
      for (int s0 = 0; s0 < cnt; s0 += kUnDepth) {
        if (k != 0 || j0 != 0 || s0 != 0) load_values(k, j0 + s0);
#pragma unroll
        for (int jj = 0; jj < kUnDepth; ++jj) {
          if (s0 + jj < cnt) {
            const float wj = wgt[k * kUnPiece + s0 + jj];
            float2& a = acc[kEntries ? (jj & 7) : 0];
            a.x = fmaf(wj, v[jj].x, a.x);
            a.y = fmaf(wj, v[jj].y, a.y);
          }
        }
      }
      if (tid == 0) add_den(k, cnt, den);  // after this thread's loads are out
    }
    float2 tot = acc[0];
    float dtot = den[0];
    if (kEntries) {
      tot = make_float2(((acc[0].x + acc[1].x) + (acc[2].x + acc[3].x)) + ((acc[4].x + acc[5].x) + (acc[6].x + acc[7].x)),
                        ((acc[0].y + acc[1].y) + (acc[2].y + acc[3].y)) + ((acc[4].y + acc[5].y) + (acc[6].y + acc[7].y)));
      dtot = ((den[0] + den[1]) + (den[2] + den[3])) + ((den[4] + den[5]) + (den[6] + den[7]));
    }
    lat2[k * (kRank / 2) + tid] = tot;
    if (tid == 0) row_den[k] = dtot;
  }
  __syncthreads();
  if (tid < nrows && p.out_lse != nullptr && vblk == 0) {
    const int rr = rr0 + tid, b = rr / p.q_len;
    p.out_lse[static_cast<long long>(b) * rows_total + row_r[tid]] = merged_lse(row_m[tid], row_den[tid]);
  }
  for (int k = 0; k < nrows; ++k) {
    const float2 a = lat2[k * (kRank / 2) + tid];
    const float den = row_den[k];
    lat2[k * (kRank / 2) + tid] = (row_m[k] == -INFINITY) ? make_float2(0.f, 0.f) : make_float2(a.x / den, a.y / den);
  }
  __syncthreads();
  // out_v[row][col] = sum_d lat[row][d] * W[d][col]: warp w sums d in [64 w, 64 w + 64) in order for each
  // real row of the group (lane = column, its 64 weights in registers), into its chunk sums; the eight
  // chunk sums are then added in chunk order.
  float* part = reinterpret_cast<float*>(smem_raw + kUnPartOff);  // [8 chunks][16 rows][32 columns]
  for (int k = 0; k < nrows; ++k) {
    const float4* lrow = reinterpret_cast<const float4*>(lat + k * kRank + w * kUnDper);
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < kUnDper / 4; ++q) {
      const float4 l4 = lrow[q];
      acc = fmaf(l4.x, wreg[4 * q + 0], acc);
      acc = fmaf(l4.y, wreg[4 * q + 1], acc);
      acc = fmaf(l4.z, wreg[4 * q + 2], acc);
      acc = fmaf(l4.w, wreg[4 * q + 3], acc);
    }
    part[(w * kUnRows + k) * kUnCols + lane] = acc;
  }
  __syncthreads();
  const int col = vblk * kUnCols + lane;
  for (int k = w; k < nrows; k += kUnChunks) {  // warp w writes rows w, w + 8
    float v = 0.f;
#pragma unroll
    for (int c = 0; c < kUnChunks; ++c) v += part[(c * kUnRows + k) * kUnCols + lane];
    const int rr = rr0 + k, b = rr / p.q_len, i = rr % p.q_len;
    const long long o = ((static_cast<long long>(b) * p.q_len + i) * p.H + h) * p.v_head + col;
    if (p.out_dtype == 2)
      static_cast<float*>(p.out)[o] = v;
    else
      static_cast<uint16_t*>(p.out)[o] = (p.out_dtype == 1) ? f2h<true>(v) : f2h<false>(v);
  }
}

}  // namespace

cudaError_t launch_cache_append(const AppendParams& p, cudaStream_t stream) {
  const long long toks = static_cast<long long>(p.B) * p.q_len;
  const long long blocks = (toks + kAppendWarps - 1) / kAppendWarps;
  if (blocks <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(kAppendWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_cache_append_kernel, p);
}

cudaError_t launch_merge_unembed(const UnembedParams& p, bool w_bf16, cudaStream_t stream) {
  static bool smem_set[4] = {false, false, false, false};
  const int inst = (w_bf16 ? 1 : 0) + (p.entries ? 2 : 0);
  const void* fns[4] = {reinterpret_cast<const void*>(&mla_merge_unembed_kernel<false, false>),
                        reinterpret_cast<const void*>(&mla_merge_unembed_kernel<true, false>),
                        reinterpret_cast<const void*>(&mla_merge_unembed_kernel<false, true>),
                        reinterpret_cast<const void*>(&mla_merge_unembed_kernel<true, true>)};
  if (!smem_set[inst]) {
    const cudaError_t e = cudaFuncSetAttribute(fns[inst], cudaFuncAttributeMaxDynamicSharedMemorySize, kUnSmem);
    if (e != cudaSuccess) return e;
    smem_set[inst] = true;
  }
  const long long R = static_cast<long long>(p.B) * p.q_len;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.H), static_cast<unsigned>(p.v_head / kUnCols),
                     static_cast<unsigned>((R + kUnRows - 1) / kUnRows));
  cfg.blockDim = dim3(kUnThreads, 1, 1);
  cfg.dynamicSmemBytes = kUnSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (inst) {
    case 0: return cudaLaunchKernelEx(&cfg, mla_merge_unembed_kernel<false, false>, p);
    case 1: return cudaLaunchKernelEx(&cfg, mla_merge_unembed_kernel<true, false>, p);
    case 2: return cudaLaunchKernelEx(&cfg, mla_merge_unembed_kernel<false, true>, p);
    default: return cudaLaunchKernelEx(&cfg, mla_merge_unembed_kernel<true, true>, p);
  }
}

cudaError_t wrap_read_clear_error(uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_device_error, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(uint32_t));
}

}  // namespace mla
