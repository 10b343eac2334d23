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
//    head) one CTA merges the rows' partials over all 512 latent columns (the
//    merge kernel's arithmetic, so the fp32 latent is the bits mla_merge_states
//    would give, never rounded), stages them and the head's W_UV^T slice
//    [512 x 32] in shared memory, and takes the product in fp32 in a fixed
//    order (d = 0 .. 511), rounded once to the output type.
#include "device_common.cuh"

namespace mla {

namespace {

constexpr int kAppendWarps = 4;

__global__ void __launch_bounds__(kAppendWarps * 32) mla_cache_append_kernel(const AppendParams p) {
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
constexpr uint32_t kUnSmem = kUnRows * kRank * 4 + kRank * kUnCols * 2;  // latent rows + W slice: 64 KB

template <bool BF16>
__global__ void __launch_bounds__(kUnThreads) mla_merge_unembed_kernel(const UnembedParams p) {
  extern __shared__ uint8_t smem_raw[];
  float* lat = reinterpret_cast<float*>(smem_raw);                          // [16][512] fp32
  uint16_t* wsl = reinterpret_cast<uint16_t*>(smem_raw + kUnRows * kRank * 4);  // [512][32] 16-bit
  pdl_wait();  // a programmatic dependent of the partial kernel: its partials are complete after this
  pdl_launch_dependents();
  const int tid = threadIdx.x;
  const int h = blockIdx.x, vblk = blockIdx.y;
  const int rows_total = p.q_len * p.H;
  const int R = p.B * p.q_len;  // rows of head h
  const int rr0 = blockIdx.z * kUnRows;
  const int nrows = min(kUnRows, R - rr0);
  // this head's W_UV^T columns [32 vblk, 32 vblk + 32): 512 rows of 64 bytes
  const uint16_t* wsrc = p.w_uv_t + (static_cast<long long>(h) * kRank) * p.v_head + vblk * kUnCols;
  for (int x = tid; x < kRank * 4; x += kUnThreads) {
    const int d = x >> 2, q = x & 3;
    reinterpret_cast<uint4*>(wsl + d * kUnCols)[q] =
        *reinterpret_cast<const uint4*>(wsrc + static_cast<long long>(d) * p.v_head + q * 8);
  }
  // the merged latent of each row (row rr of head h = query row i of request b)
  for (int x = tid; x < kUnRows * (kRank / 4) + kUnRows; x += kUnThreads) {
    const bool is_lse = x >= kUnRows * (kRank / 4);
    const int k = is_lse ? x - kUnRows * (kRank / 4) : x / (kRank / 4);
    const int c = is_lse ? 0 : (x % (kRank / 4)) * 4;
    if (k >= nrows) {
      if (!is_lse) *reinterpret_cast<float4*>(lat + k * kRank + c) = make_float4(0.f, 0.f, 0.f, 0.f);
      continue;
    }
    const int rr = rr0 + k, b = rr / p.q_len, i = rr % p.q_len;
    const int lo = __ldg(p.o_indptr + b), hi = __ldg(p.o_indptr + b + 1);
    float M, den;
    const float4 acc = merge_cols4(p.partials, p.lse, lo, hi - lo, rows_total, i * p.H + h, c, !is_lse, &M, &den);
    if (is_lse) {
      if (p.out_lse != nullptr && vblk == 0) p.out_lse[static_cast<long long>(b) * rows_total + i * p.H + h] =
          merged_lse(M, den);
    } else {
      *reinterpret_cast<float4*>(lat + k * kRank + c) = acc;
    }
  }
  __syncthreads();
  // out_v[row][col] = sum_d lat[row][d] * W[d][col], d in order; warp w takes rows w and w + 8
  const int lane = tid & 31, w = tid >> 5;
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 8
  for (int d = 0; d < kRank; ++d) {
    const float wv = h2f<BF16>(wsl[d * kUnCols + lane]);
    acc0 = fmaf(lat[w * kRank + d], wv, acc0);
    acc1 = fmaf(lat[(w + 8) * kRank + d], wv, acc1);
  }
  const int col = vblk * kUnCols + lane;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int k = w + 8 * u;
    if (k >= nrows) continue;
    const int rr = rr0 + k, b = rr / p.q_len, i = rr % p.q_len;
    const long long o = ((static_cast<long long>(b) * p.q_len + i) * p.H + h) * p.v_head + col;
    const float v = u ? acc1 : acc0;
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
  mla_cache_append_kernel<<<static_cast<unsigned>(blocks), kAppendWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_merge_unembed(const UnembedParams& p, bool w_bf16, cudaStream_t stream) {
  static bool smem_set[2] = {false, false};
  const void* fn = w_bf16 ? reinterpret_cast<const void*>(&mla_merge_unembed_kernel<true>)
                          : reinterpret_cast<const void*>(&mla_merge_unembed_kernel<false>);
  if (!smem_set[w_bf16 ? 1 : 0]) {
    const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kUnSmem);
    if (e != cudaSuccess) return e;
    smem_set[w_bf16 ? 1 : 0] = true;
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
  return w_bf16 ? cudaLaunchKernelEx(&cfg, mla_merge_unembed_kernel<true>, p)
                : cudaLaunchKernelEx(&cfg, mla_merge_unembed_kernel<false>, p);
}

cudaError_t wrap_read_clear_error(uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_device_error, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(uint32_t));
}

}  // namespace mla
