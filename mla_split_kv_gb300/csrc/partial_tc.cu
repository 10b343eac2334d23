// Tensor-core partial-decode kernel (tcgen05 + TMEM + TMA), sm_103a.
//
// Same operation as the CUDA-core kernel: for one chunk of one request, the
// normalized partial and base-2 LSE of absorbed MLA attention ("feat(core):
// matrix-absorbed MLA decode over a compressed-latent KV cache", *What
// changed*: SDPA(q_absorbed, ckv, ckv, scale, mask = scale * q_pe @ kpe^T)).
//
// Both contractions put tokens / latent columns on the MMA's M side and the
// CTA's NR query rows (heads x window rows) on N, so one MMA serves every
// head that shares a latent tile:
//   S^T[tok, row]  = [ckv | kpe][tok, 0:576] . Q^T        M=64 tokens, N=NR, K=576
//   O^T[d, row]   += ckv^T[d, tok] . P^T[tok, row]        M=128 (x4), N=NR, K=64
// A tile of 64 tokens (8 ckv boxes + 1 kpe box of 64x64, 128-byte swizzle) is
// the K-major A operand of the first product and, read MN-major, the A operand
// of the second: every latent byte leaves HBM once and is used twice from
// shared memory. S^T (double-buffered, M=64 layout: token t in TMEM lane
// 32*(t/16) + t%16) and O^T (M=128 layout) live in tensor memory.
//
// A tcgen05.mma with N <= 48 costs the same ~45 cycles whatever its size, so
// the pipeline is built to keep the single MMA-issuing thread busy: two 72 KB
// tile buffers fed by TMA with an L2 prefetch two tiles ahead, S^T and P^T
// double-buffered, and a softmax that normally needs no cross-warp exchange.
//
// Warp roles (192 threads): warps 0-3 softmax / O rescale / epilogue, warp 4
// TMA producer, warp 5 TMEM owner + MMA issuer.
//
// Online softmax in base 2 with a lazy reference max: P = 2^(s - m_ref) is
// formed against the current reference; only when some score exceeds it by
// more than 2^8 (always on the first tile) do the warps reduce the tile maxima,
// move the reference and rescale O^T and the row sums. P therefore stays
// <= 256 and the rescale pass is rare.
//
// With bf16 inputs P is carried as two bf16 terms (hi + lo, two MMAs per
// step): a single bf16 rounding of P (8-bit mantissa) would by itself leave a
// relative error near 1e-3 in the output.
#include "device_common.cuh"

namespace mla {

namespace {

constexpr int kThreads = 192;
constexpr float kRescaleTau = 8.0f;

template <int NR, bool SPLIT>
struct TcLayout {
  static constexpr uint32_t kQChunk = NR * 128;  // [NR x 64] 16-bit, swizzled
  static constexpr uint32_t kPBuf = NR * 128;    // P^T [NR x 64 tokens]
  static constexpr uint32_t kPStage = (SPLIT ? 2 : 1) * kPBuf;
  static constexpr uint32_t kOffQ = 2 * kTileBytes;
  static constexpr uint32_t kOffP = kOffQ + 9 * kQChunk;
  static constexpr uint32_t kOffSmall = kOffP + 2 * kPStage;  // P^T double-buffered
  static constexpr uint32_t kSmallBytes = 2048;
  static constexpr uint32_t kSmem = kOffSmall + kSmallBytes + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = (6 * NR <= 32)    ? 32
                                        : (6 * NR <= 64)  ? 64
                                        : (6 * NR <= 128) ? 128
                                        : (6 * NR <= 256) ? 256
                                                          : 512;
  static_assert(kSmem <= 232448, "shared memory per CTA");
};

struct TcSmall {
  uint64_t full[2], empty[2], sfull[2], sfree[2], pfull[2], drain;
  uint32_t tmem_base;
  int32_t abort_flag;
  float red[4][64];   // per-warp column maxima (rescale path) / row sums (epilogue)
  float mref[64];     // reference max per column (log2 units of the scaled score)
  float alpha[64];    // rescale factor per column
};
static_assert(sizeof(TcSmall) <= 2048, "small smem region");

__device__ __forceinline__ uint32_t tmem_lane_base(int warp) { return static_cast<uint32_t>(32 * (warp & 3)) << 16; }

// Descriptor advanced by a byte offset (start-address field, 16-byte units).
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

template <int NR, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    mla_partial_tc_kernel(const __grid_constant__ CUtensorMap tm_ckv, const __grid_constant__ CUtensorMap tm_kpe,
                          const PartialParams p) {
  constexpr bool SPLIT = BF16;
  pdl_launch_dependents();  // the merge of these partials may be scheduled now; it waits for this grid
  using Lay = TcLayout<NR, SPLIT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* tiles = smem;
  uint8_t* qs = smem + Lay::kOffQ;
  uint8_t* ps = smem + Lay::kOffP;
  TcSmall* sm = reinterpret_cast<TcSmall*>(smem + Lay::kOffSmall);
  volatile int32_t* abort_flag = &sm->abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const CtaWork w = cta_work(p, NR);
  const int ntiles = (w.sub1 - w.sub0 + kTileTokens - 1) / kTileTokens;
  const int rows_total = p.q_len * p.H;

  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm->full[b], 1);
      mbar_init(&sm->empty[b], 1);
      mbar_init(&sm->sfull[b], 1);
      mbar_init(&sm->sfree[b], 4);
      mbar_init(&sm->pfull[b], 4);
    }
    mbar_init(&sm->drain, 1);
    sm->abort_flag = 0;
    fence_mbar_init();
  }
  if (tid < 64) sm->mref[tid] = -INFINITY;
  if (warp == 5) {
    tmem_alloc(&sm->tmem_base, Lay::kTmemCols);
    tmem_relinquish();
  }
  // Q^T: NR rows x 576 columns, K-major, 9 swizzled [NR x 64] chunks
  if (warp < 4) {
    for (int idx = tid; idx < NR * (kQkDim / 8); idx += 128) {
      const int r = idx / (kQkDim / 8), k = (idx % (kQkDim / 8)) * 8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (r < w.nrows) {
        const long long row = static_cast<long long>(w.b) * rows_total + w.row0 + r;
        v = (k < kRank) ? *reinterpret_cast<const uint4*>(p.q_abs + row * kRank + k)
                        : *reinterpret_cast<const uint4*>(p.q_pe + row * kRope + (k - kRank));
      }
      *reinterpret_cast<uint4*>(qs + (k / kBoxCols) * Lay::kQChunk + sw128_offset(r, k % kBoxCols)) = v;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;

  if (warp == 4) {
    // ------------------------------------------------------------------ TMA producer
    const uint64_t pol = l2_policy_evict_first();
    if (lane == 0) {
      tma_prefetch_desc(&tm_ckv);
      tma_prefetch_desc(&tm_kpe);
    }
    const int npages_req = (w.L + p.bs - 1) / p.bs;
    int win_base = -1, win_pid = -1, issued = 0;
    // physical page of logical page pg (warp-uniform pg), through a 32-entry window
    auto page_of = [&](int pg) -> int {
      const int base = pg & ~31;
      if (base != win_base) {
        win_base = base;
        const int q = base + lane;
        win_pid = (q < npages_req && q < p.max_blocks) ? checked_page(p, w.b, q) : -1;
      }
      return __shfl_sync(0xffffffffu, win_pid, pg & 31);
    };
    auto l2_prefetch = [&](int i) {  // tile i into L2 (no smem, no barrier)
      const int tok0 = w.sub0 + i * kTileTokens;
      const int npg = (min(kTileTokens, w.sub1 - tok0) + p.bs - 1) / p.bs;
      for (int k = 0; k < npg; ++k) {
        const int pid = page_of(tok0 / p.bs + k);
        if (lane == 0 && pid >= 0) {
          for (int c = 0; c < kBoxesPerTile - 1; ++c) tma_prefetch_l2_2d(&tm_ckv, c * kBoxCols, pid * p.bs);
          tma_prefetch_l2_2d(&tm_kpe, 0, pid * p.bs);
        }
      }
    };
    for (int i = 0; i < ntiles; ++i) {
      const int buf = i & 1;
      if (i >= 2) {
        int ok = 1;
        if (lane == 0) {
          ok = mbar_wait(&sm->empty[buf], ((i >> 1) - 1) & 1, p.timeout_ns) && !*abort_flag;
          if (!ok) *abort_flag = 1;
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;  // lane 0 decides for the warp
      }
      const int tok0 = w.sub0 + i * kTileTokens;
      const int ntok = min(kTileTokens, w.sub1 - tok0);
      const int pg0 = tok0 / p.bs;
      const int npg = (ntok + p.bs - 1) / p.bs;
      int pids[kTileTokens / 16];
#pragma unroll
      for (int k = 0; k < kTileTokens / 16; ++k) pids[k] = (k < npg) ? page_of(pg0 + k) : -1;
      if (lane == 0) {
        uint8_t* tb = tiles + buf * kTileBytes;
        mbar_arrive_expect_tx(&sm->full[buf], static_cast<uint32_t>(npg * p.bs * 128 * kBoxesPerTile));
        for (int k = 0; k < npg; ++k) {
          const int y = pids[k] * p.bs;
          for (int c = 0; c < kBoxesPerTile - 1; ++c)
            tma_load_2d(tb + c * kBoxBytes + k * p.bs * 128, &tm_ckv, c * kBoxCols, y, &sm->full[buf], pol);
          tma_load_2d(tb + (kBoxesPerTile - 1) * kBoxBytes + k * p.bs * 128, &tm_kpe, 0, y, &sm->full[buf], pol);
        }
      }
      issued = i + 1;
      if (i + 2 < ntiles) l2_prefetch(i + 2);
    }
    if (lane == 0 && *abort_flag) {  // let loads in flight land before smem is released
      for (int i = (issued > 2 ? issued - 2 : 0); i < issued; ++i)
        mbar_wait(&sm->full[i & 1], (i >> 1) & 1, kDrainTimeoutNs);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------------ MMA issuer
    const uint32_t idesc_s = idesc_f16_f32(64, NR, BF16, false, false);
    const uint32_t idesc_o = idesc_f16_f32(128, NR, BF16, true, false);
    const uint32_t t_addr = smem_u32(tiles);
    const uint64_t q_desc = smem_desc_sw128(smem_u32(qs), 16, 1024);
    const uint64_t p_desc = smem_desc_sw128(smem_u32(ps), 16, 1024);
    auto issue_pv = [&](int j) -> bool {
      const int b = j & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&sm->pfull[b], (j >> 1) & 1, p.timeout_ns);
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        if (lane == 0) *abort_flag = 1;
        return false;
      }
      if (lane == 0) {
        tc_fence_after();
        const uint64_t a0 = smem_desc_sw128(t_addr + b * kTileBytes, kBoxBytes, 1024);
        const uint64_t pb = desc_add(p_desc, b * Lay::kPStage);
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t adesc = desc_add(a0, 2 * blk * kBoxBytes + ks * 16 * 128);
            umma_f16_ss(tmem + 2 * NR + blk * NR, adesc, desc_add(pb, ks * 32), idesc_o, (j > 0 || ks > 0) ? 1u : 0u);
            if constexpr (SPLIT)
              umma_f16_ss(tmem + 2 * NR + blk * NR, adesc, desc_add(pb, Lay::kPBuf + ks * 32), idesc_o, 1u);
          }
        }
        umma_commit(&sm->empty[b]);  // tile buffer b and P^T buffer b are free again
      }
      __syncwarp();
      return true;
    };
    bool alive = true;
    for (int i = 0; i < ntiles; ++i) {
      const int buf = i & 1;
      int ok = 1;
      if (lane == 0) {
        ok = mbar_wait(&sm->full[buf], (i >> 1) & 1, p.timeout_ns) && !*abort_flag;
        if (!ok) *abort_flag = 1;
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) {  // lane 0 decides for the warp
        alive = false;
        break;
      }
      const int nvalid = min(kTileTokens, w.sub1 - (w.sub0 + i * kTileTokens));
      if (nvalid < kTileTokens) {  // rows past the chunk end: zero them (finite A operand)
        uint8_t* tb = tiles + buf * kTileBytes;
        const int nz = (kTileTokens - nvalid) * 8;
        for (int c = 0; c < kBoxesPerTile; ++c)
          for (int j = lane; j < nz; j += 32)
            *reinterpret_cast<uint4*>(tb + c * kBoxBytes + nvalid * 128 + j * 16) = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (i >= 2) {
        if (lane == 0) ok = mbar_wait(&sm->sfree[buf], ((i >> 1) - 1) & 1, p.timeout_ns);
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          if (lane == 0) *abort_flag = 1;
          alive = false;
          break;
        }
      }
      if (lane == 0) {
        tc_fence_after();
        const uint64_t a0 = smem_desc_sw128(t_addr + buf * kTileBytes, 16, 1024);
#pragma unroll
        for (int c = 0; c < kBoxesPerTile; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_f16_ss(tmem + buf * NR, desc_add(a0, c * kBoxBytes + kk * 32),
                        desc_add(q_desc, c * Lay::kQChunk + kk * 32), idesc_s, (c | kk) != 0 ? 1u : 0u);
        umma_commit(&sm->sfull[buf]);
      }
      __syncwarp();
      if (i >= 1 && !issue_pv(i - 1)) {
        alive = false;
        break;
      }
    }
    if (alive && ntiles >= 1) issue_pv(ntiles - 1);
    if (lane == 0) {  // every MMA issued so far has completed before TMEM is read or freed
      umma_commit(&sm->drain);
      mbar_wait(&sm->drain, 0, kDrainTimeoutNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax (warps 0-3)
    // Thread (warp, lane < 16) owns token 16*warp + lane of each tile (M=64 layout of S^T).
    float lsum[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) lsum[r] = 0.f;
    const bool owns_token = lane < 16;
    const int tl = 16 * warp + lane;
    // smallest causal limit over this CTA's rows: tiles below it need no causal mask
    const int causal_floor = p.causal ? w.L - p.q_len + w.row0 / p.H : 0x7fffffff;
    for (int i = 0; i < ntiles; ++i) {
      const int buf = i & 1;
      const int tok0 = w.sub0 + i * kTileTokens;
      const int nvalid = min(kTileTokens, w.sub1 - tok0);
      const bool masked_tile = (nvalid < kTileTokens) || (tok0 + kTileTokens - 1 > causal_floor) ||
                               (w.nrows < NR);
      float x[NR];
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&sm->sfull[buf], (i >> 1) & 1, p.timeout_ns);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      bool need_local = false;
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < NR; c += 16) tmem_ld16(tmem + tmem_lane_base(warp) + buf * NR + c, x + c);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->sfree[buf]);
        const int t = tok0 + tl;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          bool vis = owns_token;
          if (masked_tile) {
            vis = vis && (tl < nvalid) && (r < w.nrows);
            if (p.causal) vis = vis && (t <= w.L - p.q_len + (w.row0 + r) / p.H);
          }
          x[r] = vis ? x[r] * p.scale_log2 : -INFINITY;
          need_local |= x[r] > sm->mref[r] + kRescaleTau;
        }
      } else {
#pragma unroll
        for (int r = 0; r < NR; ++r) x[r] = -INFINITY;
        if (lane == 0) *abort_flag = 1;
      }
      // one barrier per tile; it is also where an abort becomes a uniform decision
      if (named_bar_sync_or(1, 128, need_local || *abort_flag != 0)) {
        if (named_bar_sync_or(1, 128, *abort_flag != 0)) break;
        // rare path: move the reference max, rescale O^T and the row sums
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          float v = x[r];
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
          if (lane == 0) sm->red[warp][r] = v;
        }
        named_bar_sync(1, 128);
        if (tid < NR) {
          const float mprev = sm->mref[tid];
          const float tmax = fmaxf(fmaxf(sm->red[0][tid], sm->red[1][tid]), fmaxf(sm->red[2][tid], sm->red[3][tid]));
          const float mnew = fmaxf(mprev, tmax);
          sm->alpha[tid] = (mnew == -INFINITY) ? 1.f : exp2f(mprev - mnew);
          sm->mref[tid] = mnew;
        }
        named_bar_sync(1, 128);
        if (i >= 1) {  // PV(i-1) must be complete before O^T is rescaled
          int ok2 = 1;
          if (lane == 0) ok2 = mbar_wait(&sm->empty[(i - 1) & 1], ((i - 1) >> 1) & 1, p.timeout_ns);
          if (__shfl_sync(0xffffffffu, ok2, 0)) {
            tc_fence_after();
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
#pragma unroll
              for (int c = 0; c < NR; c += 16) {
                float v[16];
                const uint32_t a = tmem + tmem_lane_base(warp) + 2 * NR + blk * NR + c;
                tmem_ld16(a, v);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] *= sm->alpha[c + j];
                tmem_st16(a, v);
              }
            }
            tmem_wait_st();
          } else if (lane == 0) {
            *abort_flag = 1;
          }
        }
#pragma unroll
        for (int r = 0; r < NR; ++r) lsum[r] *= sm->alpha[r];
      }
      // P^T buffer `buf` was last read by PV(i-2)
      if (i >= 2) {
        int ok3 = 1;
        if (lane == 0) ok3 = mbar_wait(&sm->empty[buf], ((i >> 1) - 1) & 1, p.timeout_ns);
        if (!__shfl_sync(0xffffffffu, ok3, 0) && lane == 0) *abort_flag = 1;
      }
      if (owns_token) {  // probabilities -> P^T (16-bit, K-major, swizzled) and row sums
        uint8_t* pb = ps + buf * Lay::kPStage;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          const float pr = (x[r] == -INFINITY) ? 0.f : exp2f(x[r] - sm->mref[r]);
          const uint16_t hv = f2h<BF16>(pr);
          float used = h2f<BF16>(hv);
          *reinterpret_cast<uint16_t*>(pb + sw128_offset(r, tl)) = hv;
          if constexpr (SPLIT) {
            const uint16_t lv = f2h<BF16>(pr - used);
            used += h2f<BF16>(lv);
            *reinterpret_cast<uint16_t*>(pb + Lay::kPBuf + sw128_offset(r, tl)) = lv;
          }
          lsum[r] += used;
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->pfull[buf]);
    }
    // after the last PV: reduce the row sums over the 64 token lanes
    const bool aborted = named_bar_sync_or(1, 128, *abort_flag != 0);  // same answer in all 4 warps
    if (ntiles > 0 && !aborted) {
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&sm->empty[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, p.timeout_ns);
      if (!__shfl_sync(0xffffffffu, ok, 0) && lane == 0) *abort_flag = 1;
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      float v = owns_token ? lsum[r] : 0.f;
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      if (lane == 0) sm->red[warp][r] = v;
    }
    named_bar_sync(1, 128);
  }
  __syncthreads();  // all roles done: tiles are free for staging
  const bool have = (ntiles > 0) && !*abort_flag;
  float* ostage = reinterpret_cast<float*>(tiles);  // [NR][512]
  float* mst = ostage + NR * kRank;
  float* lst = mst + NR;
  if (warp < 4) {
    if (have) {
      tc_fence_after();
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
#pragma unroll
        for (int c = 0; c < NR; c += 16) {
          float v[16];
          tmem_ld16(tmem + tmem_lane_base(warp) + 2 * NR + blk * NR + c, v);
          tmem_wait_ld();
          const int d = blk * 128 + warp * 32 + lane;
#pragma unroll
          for (int j = 0; j < 16; ++j) ostage[(c + j) * kRank + d] = v[j];
        }
      }
    } else {
      for (int idx = tid; idx < NR * kRank; idx += 128) ostage[idx] = 0.f;
    }
    if (tid < NR) {
      mst[tid] = have ? sm->mref[tid] : -INFINITY;
      lst[tid] = have ? (sm->red[0][tid] + sm->red[1][tid]) + (sm->red[2][tid] + sm->red[3][tid]) : 0.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  cluster_combine(p, w, ostage, mst, lst, tid, kThreads);
  cluster_sync();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::kTmemCols);
  }
}

template <int NR, bool BF16>
const void* tc_fn() {
  return reinterpret_cast<const void*>(&mla_partial_tc_kernel<NR, BF16>);
}

// Instantiated variants: {16, 32, 48} rows for fp16 and bf16 (64 rows would not
// fit next to two 72 KB tiles once P^T is double-buffered).
const void* tc_kernel_ptr(int nr, bool bf16) {
  switch (nr) {
    case 16: return bf16 ? tc_fn<16, true>() : tc_fn<16, false>();
    case 32: return bf16 ? tc_fn<32, true>() : tc_fn<32, false>();
    default: return bf16 ? tc_fn<48, true>() : tc_fn<48, false>();
  }
}

uint32_t tc_smem(int nr, bool bf16) {
  switch (nr) {
    case 16: return bf16 ? TcLayout<16, true>::kSmem : TcLayout<16, false>::kSmem;
    case 32: return bf16 ? TcLayout<32, true>::kSmem : TcLayout<32, false>::kSmem;
    default: return bf16 ? TcLayout<48, true>::kSmem : TcLayout<48, false>::kSmem;
  }
}

int variant_index(int nr, bool bf16) { return (bf16 ? 3 : 0) + (nr == 16 ? 0 : (nr == 32 ? 1 : 2)); }

// Kernel attributes, set once per variant.
cudaError_t prepare(const void* fn, int nr, bool bf16, int cluster) {
  static bool smem_set[6] = {false, false, false, false, false, false};
  static bool np_set[6] = {false, false, false, false, false, false};
  const int v = variant_index(nr, bf16);
  cudaError_t e = cudaSuccess;
  if (!smem_set[v]) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, tc_smem(nr, bf16));
    if (e != cudaSuccess) return e;
    smem_set[v] = true;
  }
  if (cluster > 8 && !np_set[v]) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    np_set[v] = true;
  }
  return e;
}

}  // namespace

// Rows per CTA: the fewest groups of at most 48 rows, balanced, rounded up to 16.
int tc_rows_per_cta(int total_rows, bool) {
  const int groups = (total_rows + 47) / 48;
  const int per = (total_rows + groups - 1) / groups;
  return per <= 16 ? 16 : (per <= 32 ? 32 : 48);
}

cudaError_t launch_partial_tc(const CUtensorMap& tm_ckv, const CUtensorMap& tm_kpe, const CUtensorMap& tm_pages,
                              const CUtensorMap& tm_kpe_half, const PartialParams& p, int num_chunks, int cluster,
                              bool bf16, cudaStream_t stream) {
  const int rows = p.q_len * p.H;
  if (tc128_supports(rows, bf16, cluster))
    return launch_partial_tc128(tm_pages, tm_kpe_half, p, num_chunks, cluster, bf16, stream);
  if (mh_supports(rows, cluster))
    return (p.xchg16 == 2) ? launch_partial_mh_nx(tm_pages, tm_kpe_half, p, num_chunks, bf16, stream)
                           : launch_partial_mh(tm_pages, tm_kpe_half, p, num_chunks, bf16, stream);
  const int nr = tc_rows_per_cta(rows, bf16);
  const void* fn = tc_kernel_ptr(nr, bf16);
  cudaError_t e = prepare(fn, nr, bf16, cluster);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster, num_chunks, (rows + nr - 1) / nr);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = tc_smem(nr, bf16);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bf16) {
    switch (nr) {
      case 16: return cudaLaunchKernelEx(&cfg, mla_partial_tc_kernel<16, true>, tm_ckv, tm_kpe, p);
      case 32: return cudaLaunchKernelEx(&cfg, mla_partial_tc_kernel<32, true>, tm_ckv, tm_kpe, p);
      default: return cudaLaunchKernelEx(&cfg, mla_partial_tc_kernel<48, true>, tm_ckv, tm_kpe, p);
    }
  }
  switch (nr) {
    case 16: return cudaLaunchKernelEx(&cfg, mla_partial_tc_kernel<16, false>, tm_ckv, tm_kpe, p);
    case 32: return cudaLaunchKernelEx(&cfg, mla_partial_tc_kernel<32, false>, tm_ckv, tm_kpe, p);
    default: return cudaLaunchKernelEx(&cfg, mla_partial_tc_kernel<48, false>, tm_ckv, tm_kpe, p);
  }
}

int tc_max_active_clusters(int cluster, int rows_per_cta, bool bf16) {
  const void* fn = tc_kernel_ptr(rows_per_cta, bf16);
  if (prepare(fn, rows_per_cta, bf16, cluster) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = tc_smem(rows_per_cta, bf16);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t tc_read_clear_error(uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_device_error, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(uint32_t));
}

}  // namespace mla
