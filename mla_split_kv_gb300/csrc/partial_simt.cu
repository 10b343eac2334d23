// CUDA-core partial-decode kernel: fp32 FMA on 16 query rows per CTA.
//
// Computes, for one chunk of one request, the normalized partial and base-2
// LSE of absorbed MLA attention ("feat(core): matrix-absorbed MLA decode over
// a compressed-latent KV cache", *What changed*, Stage 1 / Stage 2): scores
// s = scale*(q_abs . ckv + q_pe . kpe), softmax over the chunk, weighted sum
// of ckv rows. The latent tile is staged by TMA (two 72 KB buffers of 64
// tokens x [512 | 64] columns, 128-byte swizzled) and consumed by all 256
// threads with fp32 FMA. The CTAs of a cluster split the chunk and combine
// their (max, sum, O) through distributed shared memory in rank order.
#include "device_common.cuh"

namespace mla {

namespace {

constexpr int kThreads = 256;
constexpr int kRows = 16;                 // query rows per CTA
constexpr int kQStride = kQkDim + 4;      // padded fp32 row of the query copy
constexpr uint32_t kOffQ = 2 * kTileBytes;
constexpr uint32_t kOffP = kOffQ + kRows * kQStride * 4;   // probabilities [64][16]
constexpr uint32_t kOffRed = kOffP + kTileTokens * kRows * 4;
constexpr uint32_t kOffBar = kOffRed + 2 * 8 * kRows * 4;  // two [8 warps][16] arrays
constexpr uint32_t kSmemBytes = kOffBar + 64 + 1024;      // + alignment slack

template <bool BF16>
__device__ __forceinline__ void unpack8(uint4 raw, float* f) {
  const uint16_t* h = reinterpret_cast<const uint16_t*>(&raw);
#pragma unroll
  for (int j = 0; j < 8; ++j) f[j] = h2f<BF16>(h[j]);
}

// Issue the TMA loads of tile i (pages of the request) into buffer i % 2.
__device__ __forceinline__ void issue_tile(const PartialParams& p, const CtaWork& w, int i, uint8_t* tiles,
                                           uint64_t* full, const CUtensorMap* tm_ckv, const CUtensorMap* tm_kpe,
                                           uint64_t pol) {
  const int buf = i & 1;
  const int tok0 = w.sub0 + i * kTileTokens;
  const int ntok = min(kTileTokens, w.sub1 - tok0);
  const int pg0 = tok0 / p.bs;
  const int npg = (ntok + p.bs - 1) / p.bs;
  uint8_t* tb = tiles + buf * kTileBytes;
  mbar_arrive_expect_tx(&full[buf], static_cast<uint32_t>(npg * p.bs * 128 * kBoxesPerTile));
  for (int k = 0; k < npg; ++k) {
    int pid = -1;
    if (pg0 + k < p.max_blocks) pid = checked_page(p, w.b, pg0 + k);
    const int y = pid * p.bs;
    for (int c = 0; c < kBoxesPerTile - 1; ++c)
      tma_load_2d(tb + c * kBoxBytes + k * p.bs * 128, tm_ckv, c * kBoxCols, y, &full[buf], pol);
    tma_load_2d(tb + (kBoxesPerTile - 1) * kBoxBytes + k * p.bs * 128, tm_kpe, 0, y, &full[buf], pol);
  }
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    mla_partial_simt_kernel(const __grid_constant__ CUtensorMap tm_ckv, const __grid_constant__ CUtensorMap tm_kpe,
                            const PartialParams p) {
  extern __shared__ uint8_t smem_raw[];
  pdl_launch_dependents();  // the merge of these partials may be scheduled now; it waits for this grid
  uint8_t* smem = align1024(smem_raw);
  uint8_t* tiles = smem;
  float* qs = reinterpret_cast<float*>(smem + kOffQ);
  float* ps = reinterpret_cast<float*>(smem + kOffP);
  float* red_max = reinterpret_cast<float*>(smem + kOffRed);
  float* red_sum = red_max + 8 * kRows;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + kOffBar + 16);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const CtaWork w = cta_work(p, kRows);
  const int ntiles = (w.sub1 - w.sub0 + kTileTokens - 1) / kTileTokens;
  const int rows_total = p.q_len * p.H;

  // query rows as fp32 (rows past the end are zero)
  for (int idx = tid; idx < kRows * (kQkDim / 8); idx += kThreads) {
    const int r = idx / (kQkDim / 8), k = (idx % (kQkDim / 8)) * 8;
    float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (r < w.nrows) {
      const long long row = static_cast<long long>(w.b) * rows_total + w.row0 + r;
      const uint4 raw = (k < kRank) ? *reinterpret_cast<const uint4*>(p.q_abs + row * kRank + k)
                                    : *reinterpret_cast<const uint4*>(p.q_pe + row * kRope + (k - kRank));
      unpack8<BF16>(raw, f);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) qs[r * kQStride + k + j] = f[j];
  }
  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const uint64_t pol = l2_policy_evict_first();
  if (tid == 0) {
    tma_prefetch_desc(&tm_ckv);
    tma_prefetch_desc(&tm_kpe);
    for (int i = 0; i < 2 && i < ntiles; ++i) issue_tile(p, w, i, tiles, full, &tm_ckv, &tm_kpe, pol);
  }

  // per-thread state: O[16 rows][2 columns d0, d0+1]; m and l replicated
  float o[kRows][2];
  float m[kRows], l[kRows];
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    o[r][0] = o[r][1] = 0.f;
    m[r] = -INFINITY;
    l[r] = 0.f;
  }
  const int d0 = 2 * tid;  // PV columns of this thread
  const int pv_box = d0 >> 6, pv_col = d0 & 63;
  // QK mapping: token tl of the tile, rows rg, rg+4, rg+8, rg+12 (the four
  // row groups of a warp hit distinct shared-memory banks)
  const int tl = 8 * warp + (lane & 7);
  const int rg = lane >> 3;

  int issued = ntiles < 2 ? ntiles : 2;
  for (int i = 0; i < ntiles; ++i) {
    const int buf = i & 1;
    bool ok = true;
    if (tid == 0) ok = mbar_wait(&full[buf], (i >> 1) & 1, p.timeout_ns);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) *abort_flag = 1;
      break;
    }
    const uint8_t* tb = tiles + buf * kTileBytes;
    const int tok0 = w.sub0 + i * kTileTokens;
    const int nvalid = min(kTileTokens, w.sub1 - tok0);

    // --- scores: 4 rows x 1 token per thread, fp32 FMA over 576 dims
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
    for (int c = 0; c < kQkDim / 8; ++c) {
      const int box = c >> 3, col = (c & 7) * 8;
      const uint4 raw = *reinterpret_cast<const uint4*>(tb + box * kBoxBytes + sw128_offset(tl, col));
      float kf[8];
      unpack8<BF16>(raw, kf);
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const float4 qa = *reinterpret_cast<const float4*>(qs + (rg + 4 * rr) * kQStride + c * 8);
        const float4 qb = *reinterpret_cast<const float4*>(qs + (rg + 4 * rr) * kQStride + c * 8 + 4);
        acc[rr] = fmaf(qa.x, kf[0], acc[rr]);
        acc[rr] = fmaf(qa.y, kf[1], acc[rr]);
        acc[rr] = fmaf(qa.z, kf[2], acc[rr]);
        acc[rr] = fmaf(qa.w, kf[3], acc[rr]);
        acc[rr] = fmaf(qb.x, kf[4], acc[rr]);
        acc[rr] = fmaf(qb.y, kf[5], acc[rr]);
        acc[rr] = fmaf(qb.z, kf[6], acc[rr]);
        acc[rr] = fmaf(qb.w, kf[7], acc[rr]);
      }
    }
    const int t = tok0 + tl;
    float x[4];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int r = rg + 4 * rr;
      const int row = w.row0 + r;
      bool vis = (tl < nvalid) && (r < w.nrows);
      if (p.causal) vis = vis && (t <= w.L - p.q_len + row / p.H);
      x[rr] = vis ? acc[rr] * p.scale_log2 : -INFINITY;
      float mx = x[rr];
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      if ((lane & 7) == 0) red_max[warp * kRows + r] = mx;
    }
    __syncthreads();
    // new running max (replicated in every thread) and the rescale factors
    float alpha[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      float tmax = red_max[r];
#pragma unroll
      for (int k = 1; k < 8; ++k) tmax = fmaxf(tmax, red_max[k * kRows + r]);
      const float mn = fmaxf(m[r], tmax);
      alpha[r] = (mn == -INFINITY) ? 1.f : exp2f(m[r] - mn);
      m[r] = mn;
    }
    // probabilities of this thread's token, their partial sums
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int r = rg + 4 * rr;
      const float pr = (x[rr] == -INFINITY) ? 0.f : exp2f(x[rr] - m[r]);
      ps[tl * kRows + r] = pr;
      float s = pr;
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      s += __shfl_xor_sync(0xffffffffu, s, 4);
      if ((lane & 7) == 0) red_sum[warp * kRows + r] = s;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      float s = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) s += red_sum[k * kRows + r];
      l[r] = l[r] * alpha[r] + s;
      o[r][0] *= alpha[r];
      o[r][1] *= alpha[r];
    }
    // --- values: O[r][d0..d0+1] += p[t][r] * ckv[t][d0..d0+1]
    for (int tt = 0; tt < nvalid; ++tt) {
      const uint32_t pair = *reinterpret_cast<const uint32_t*>(tb + pv_box * kBoxBytes + sw128_offset(tt, pv_col));
      const float v0 = h2f<BF16>(static_cast<uint16_t>(pair & 0xFFFFu));
      const float v1 = h2f<BF16>(static_cast<uint16_t>(pair >> 16));
      const float4* pp = reinterpret_cast<const float4*>(ps + tt * kRows);
#pragma unroll
      for (int q4 = 0; q4 < kRows / 4; ++q4) {
        const float4 pr = pp[q4];
        o[q4 * 4 + 0][0] = fmaf(pr.x, v0, o[q4 * 4 + 0][0]);
        o[q4 * 4 + 0][1] = fmaf(pr.x, v1, o[q4 * 4 + 0][1]);
        o[q4 * 4 + 1][0] = fmaf(pr.y, v0, o[q4 * 4 + 1][0]);
        o[q4 * 4 + 1][1] = fmaf(pr.y, v1, o[q4 * 4 + 1][1]);
        o[q4 * 4 + 2][0] = fmaf(pr.z, v0, o[q4 * 4 + 2][0]);
        o[q4 * 4 + 2][1] = fmaf(pr.z, v1, o[q4 * 4 + 2][1]);
        o[q4 * 4 + 3][0] = fmaf(pr.w, v0, o[q4 * 4 + 3][0]);
        o[q4 * 4 + 3][1] = fmaf(pr.w, v1, o[q4 * 4 + 3][1]);
      }
    }
    __syncthreads();  // buffer `buf`, ps and the reductions are free again
    if (tid == 0 && i + 2 < ntiles) {
      issue_tile(p, w, i + 2, tiles, full, &tm_ckv, &tm_kpe, pol);
      issued = i + 3;
    }
  }
  // after an abort, let the loads already in flight land before the buffers go away
  if (tid == 0 && *abort_flag) {
    for (int i = (issued > 2 ? issued - 2 : 0); i < issued; ++i) mbar_wait(&full[i & 1], (i >> 1) & 1, kDrainTimeoutNs);
  }
  __syncthreads();

  // --- stage (O, m, l) for the cluster combine; reuses tile buffer 0
  float* ostage = reinterpret_cast<float*>(tiles);  // [16][512]
  float* mst = ostage + kRows * kRank;
  float* lst = mst + kRows;
  const bool have = (ntiles > 0) && !*abort_flag;
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    ostage[r * kRank + d0] = have ? o[r][0] : 0.f;
    ostage[r * kRank + d0 + 1] = have ? o[r][1] : 0.f;
  }
  if (tid < kRows) {
    mst[tid] = have ? m[tid] : -INFINITY;
    lst[tid] = have ? l[tid] : 0.f;
  }
  __syncthreads();
  cluster_sync();
  cluster_combine(p, w, ostage, mst, lst, tid, kThreads);
  cluster_sync();
}

}  // namespace

int simt_rows_per_cta() { return kRows; }

cudaError_t launch_partial_simt(const CUtensorMap& tm_ckv, const CUtensorMap& tm_kpe, const PartialParams& p,
                                int num_chunks, int cluster, bool bf16, cudaStream_t stream) {
  const void* fn = bf16 ? reinterpret_cast<const void*>(&mla_partial_simt_kernel<true>)
                        : reinterpret_cast<const void*>(&mla_partial_simt_kernel<false>);
  static bool prepared[2] = {false, false};
  static bool nonportable[2] = {false, false};
  cudaError_t e = cudaSuccess;
  if (!prepared[bf16]) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    prepared[bf16] = true;
  }
  if (cluster > 8 && !nonportable[bf16]) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    nonportable[bf16] = true;
  }
  const int rows = p.q_len * p.H;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster, num_chunks, (rows + kRows - 1) / kRows);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bf16) return cudaLaunchKernelEx(&cfg, mla_partial_simt_kernel<true>, tm_ckv, tm_kpe, p);
  return cudaLaunchKernelEx(&cfg, mla_partial_simt_kernel<false>, tm_ckv, tm_kpe, p);
}

cudaError_t simt_read_clear_error(uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_device_error, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(uint32_t));
}

}  // namespace mla
