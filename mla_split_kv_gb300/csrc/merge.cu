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

// The merge of the paired kernel's pair entries into the output (mla_decode's default on that
// kernel). Entry e holds one CTA pair's unnormalized O (its tokens, all 512 columns: each CTA of
// the pair wrote its 256), its row maximum m_e and its row sum l_e relative to m_e. Per (request,
// row): M = max_e m_e, w_e = 2^(m_e - M) (0 for m_e = -inf), out = sum_e w_e O_e / sum_e w_e l_e,
// out_lse = M + log2 sum_e w_e l_e -- the merge of the pages' contract, applied to unnormalized
// parts. One warp per (request, row, 16 columns): lane = 4 g + q takes column quad q of the entries
// g, g + 8, g + 16, ... (up to 12 per lane, 96 entries, in one round of loads), sums them in entry
// order, and the warp adds the eight entry groups with a fixed shuffle tree, so the result is the
// same bits on every call.
//
// Residency: a CTA is 128 threads of at most 128 registers and no shared memory, so one fits on an
// SM beside a CTA of the paired kernel (384 threads x 128 registers, 226 KB). The merge of call n
// is therefore resident while its partial kernel runs, and it releases its own dependent (the next
// call's partial kernel) at once: that kernel waits for this one to complete before it reads
// anything, and its CTAs take each SM as the partial CTA there leaves, beside this merge's CTA.
constexpr int kEntryWarps = 4;
constexpr int kEntryGroups = 8;                  // entry groups per warp
constexpr int kEntriesPerLane = 12;              // per round of loads
constexpr int kEntryRound = kEntryGroups * kEntriesPerLane;

__global__ void __launch_bounds__(kEntryWarps * 32, 4) mla_merge_entries_kernel(const EntryMergeParams p) {
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long gw = static_cast<long long>(blockIdx.x) * kEntryWarps + warp;
  const bool active = gw < static_cast<long long>(p.B) * p.rows * 32;
  const int cb = static_cast<int>(gw & 31);  // columns [16 cb, 16 cb + 16)
  const long long br = gw >> 5;              // b * rows + row
  const int b = static_cast<int>(br / p.rows), row = static_cast<int>(br % p.rows);
  // the offsets are an input of the call, not data of the partial kernel: with tables_ready (complete
  // before that kernel started) they are read before the wait, so the entries' loads follow it at once
  int e0 = 0, e1 = 0;
  if (active && p.tables_ready) {
    e0 = __ldg(p.o_indptr + b) * p.epc;
    e1 = __ldg(p.o_indptr + b + 1) * p.epc;
  }
  pdl_wait();  // the entries are complete once the partial kernel has
  if (!active) return;
  if (!p.tables_ready) {
    e0 = p.o_indptr[b] * p.epc;
    e1 = p.o_indptr[b + 1] * p.epc;
  }
  const int g = lane >> 2, q = lane & 3;
  const int col = 16 * cb + 4 * q;
  const long long ostride = static_cast<long long>(p.rows) * kRank;  // one entry's O
  const float* const obase = p.ws_partials + static_cast<long long>(row) * kRank + col;
  const float* const mlbase = p.ws_lse + static_cast<long long>(row) * 2;  // copy 0 of the entry's m, l
  const long long mlstride = 4LL * p.rows;                                  // one entry's two copies
  // round 0: the first 96 entries' m, l and values (the values do not depend on the weights)
  float2 ml0[kEntriesPerLane];
  float4 v0[kEntriesPerLane];
#pragma unroll
  for (int j = 0; j < kEntriesPerLane; ++j) {
    const int e = e0 + g + kEntryGroups * j;
    const bool in = e < e1;
    ml0[j] = in ? __ldcg(reinterpret_cast<const float2*>(mlbase + e * mlstride)) : make_float2(-INFINITY, 0.f);
    v0[j] = in ? __ldcg(reinterpret_cast<const float4*>(obase + e * ostride)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float M = -INFINITY;
#pragma unroll
  for (int j = 0; j < kEntriesPerLane; ++j) M = fmaxf(M, ml0[j].x);
  for (int base = e0 + kEntryRound; base < e1; base += kEntryRound)
#pragma unroll
    for (int j = 0; j < kEntriesPerLane; ++j) {
      const int e = base + g + kEntryGroups * j;
      if (e < e1) M = fmaxf(M, __ldcg(mlbase + e * mlstride));
    }
  M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 4));
  M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 8));
  M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 16));
  float den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int base = e0; base < e1; base += kEntryRound) {
#pragma unroll
      for (int j = 0; j < kEntriesPerLane; ++j) {
        const int e = base + g + kEntryGroups * j;
        float2 ml;
        float4 v;
        if (base == e0) {
          ml = ml0[j];
          v = v0[j];
        } else {
          const bool in = e < e1;
          ml = in ? __ldcg(reinterpret_cast<const float2*>(mlbase + e * mlstride)) : make_float2(-INFINITY, 0.f);
          v = in ? __ldcg(reinterpret_cast<const float4*>(obase + e * ostride)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const float w = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - M);
        den = fmaf(w, ml.y, den);
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
      }
    }
  }
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    den += __shfl_xor_sync(0xffffffffu, den, o);
    acc.x += __shfl_xor_sync(0xffffffffu, acc.x, o);
    acc.y += __shfl_xor_sync(0xffffffffu, acc.y, o);
    acc.z += __shfl_xor_sync(0xffffffffu, acc.z, o);
    acc.w += __shfl_xor_sync(0xffffffffu, acc.w, o);
  }
  if (g != 0) return;
  float4 out = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) out = make_float4(acc.x / den, acc.y / den, acc.z / den, acc.w / den);
  store_out4(p.out, p.out_dtype, br * kRank + col, out);
  if (p.out_lse != nullptr && cb == 0 && q == 0) p.out_lse[br] = merged_lse(M, den);
}

}  // namespace

cudaError_t launch_merge_entries(const EntryMergeParams& p, cudaStream_t stream) {
  const long long warps = static_cast<long long>(p.B) * p.rows * 32;
  const long long blocks = (warps + kEntryWarps - 1) / kEntryWarps;
  if (blocks <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(kEntryWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_merge_entries_kernel, p);
}

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
