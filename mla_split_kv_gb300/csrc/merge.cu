// LSE-weighted merge of request-major partials (base-2 LSE).
//
// "feat(core): matrix-absorbed MLA decode over a compressed-latent KV cache",
// *How #898's merge kernel is reused*: partials of request b are rows
// o_indptr[b] .. o_indptr[b+1]-1, their LSE is base 2. "[kernel] Wire MLA
// split-KV decode", *What changed*: the reduce combines slices by their LSE so
// the result equals ordinary attention. MTPLX PR #639 commit log: a partial with
// LSE = -inf has weight 0, an all -inf row merges to zeros, and the fp32
// result is rounded once to the output dtype.
//
// One warp per (request, row, 128-column quarter); each lane owns 4 columns.
// The kernel is a programmatic dependent launch: it may be scheduled while the
// partial kernel that precedes it still runs, and waits for that grid before
// its first read, so its launch latency hides behind the partial kernel's end.
// The weights are computed lane-parallel (lane s holds partial s), the sum over
// partials runs in fixed order, so the result is bitwise reproducible.
#include "device_common.cuh"

namespace mla {

namespace {

constexpr int kWarps = 2;

__global__ void __launch_bounds__(kWarps * 32) mla_merge_kernel(const MergeParams p) {
  // Launched as a programmatic dependent of the partial kernel: everything this
  // kernel reads may still be in flight until the wait returns. The next kernel
  // (the next layer's partial kernel) is released after the wait and may start
  // its set-up while this one works.
  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long gw = static_cast<long long>(blockIdx.x) * kWarps + warp;
  const long long total = static_cast<long long>(p.B) * p.rows * 4;
  if (gw >= total) return;
  const int quarter = static_cast<int>(gw & 3);
  const long long br = gw >> 2;  // b * rows + row
  const int b = static_cast<int>(br / p.rows);
  const int row = static_cast<int>(br % p.rows);
  const int lo = p.o_indptr[b], hi = p.o_indptr[b + 1];
  const int n = hi - lo;

  const float* col = p.partials + static_cast<long long>(row) * kRank + quarter * 128 + lane * 4;
  const long long stride = static_cast<long long>(p.rows) * kRank;  // one partial slot
  // the first 8 partials' values do not depend on the weights: their loads go out with the LSE loads
  float4 v0[8];
#pragma unroll
  for (int jj = 0; jj < 8; ++jj)
    v0[jj] = (jj < n) ? *reinterpret_cast<const float4*>(col + (lo + jj) * stride) : make_float4(0.f, 0.f, 0.f, 0.f);
  // maximum LSE over this row's partials; lane s keeps the LSE of partial s (s < 32)
  const float l0 = (lane < n) ? p.lse[static_cast<long long>(lo + lane) * p.rows + row] : -INFINITY;
  float M = l0;
  for (int s = lane + 32; s < n; s += 32) M = fmaxf(M, p.lse[static_cast<long long>(lo + s) * p.rows + row]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  if (M != -INFINITY) {
    for (int s0 = 0; s0 < n; s0 += 32) {
      const int cnt = min(32, n - s0);
      float wl = 0.f;
      if (lane < cnt) {
        const float l = (s0 == 0) ? l0 : p.lse[static_cast<long long>(lo + s0 + lane) * p.rows + row];
        wl = (l == -INFINITY) ? 0.f : exp2f(l - M);
      }
      // batches of 8 partials: all loads of a batch in flight at once, then the
      // weighted sum in partial order
      for (int j0 = 0; j0 < cnt; j0 += 8) {
        float4 v[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
          v[jj] = (s0 + j0 == 0) ? v0[jj]
                  : (j0 + jj < cnt) ? *reinterpret_cast<const float4*>(col + (lo + s0 + j0 + jj) * stride)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const float wj = __shfl_sync(0xffffffffu, wl, (j0 + jj) & 31);
          if (j0 + jj < cnt) {
            den += wj;
            acc.x = fmaf(wj, v[jj].x, acc.x);
            acc.y = fmaf(wj, v[jj].y, acc.y);
            acc.z = fmaf(wj, v[jj].z, acc.z);
            acc.w = fmaf(wj, v[jj].w, acc.w);
          }
        }
      }
    }
    acc = make_float4(acc.x / den, acc.y / den, acc.z / den, acc.w / den);
  }
  const long long o_off = br * kRank + quarter * 128 + lane * 4;
  if (p.out_dtype == 2) {
    *reinterpret_cast<float4*>(static_cast<float*>(p.out) + o_off) = acc;
  } else {
    uint16_t h[4];
    const bool bf = (p.out_dtype == 1);
    const float f[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = bf ? f2h<true>(f[j]) : f2h<false>(f[j]);
    uint2 packed;
    packed.x = static_cast<uint32_t>(h[0]) | (static_cast<uint32_t>(h[1]) << 16);
    packed.y = static_cast<uint32_t>(h[2]) | (static_cast<uint32_t>(h[3]) << 16);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + o_off) = packed;
  }
  if (p.out_lse != nullptr && quarter == 0 && lane == 0)
    p.out_lse[br] = (M == -INFINITY) ? -INFINITY : M + log2f(den);
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream) {
  const long long warps = static_cast<long long>(p.B) * p.rows * 4;
  const long long blocks = (warps + kWarps - 1) / kWarps;
  if (blocks <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(kWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_merge_kernel, p);
}

}  // namespace mla
