// Tensor-core partial-decode kernel for groups of 128 query rows without a
// score exchange (score_exchange = MLA_SCORE_EXCHANGE_NONE), sm_103a.
//
// The operation is the one of the other partial kernels ("feat(core):
// matrix-absorbed MLA decode over a compressed-latent KV cache", *What
// changed*: SDPA(q_absorbed, ckv, ckv, scale, mask = scale * q_pe @ kpe^T),
// each chunk yielding a normalized partial and its log2 LSE).
//
// As in the 128-row kernel the rows sit on the MMA's M side and the two CTAs
// of a cluster pair split O's latent columns (O for 128 rows x 512 columns
// would fill all of tensor memory): CTA `half` accumulates
//   O[row, d] += P[row, tok] . ckv[tok, d]    d in [256 half, 256 half + 256)
// But each CTA computes the FULL scores
//   S[row, tok] = Q[row, :] . [ckv | kpe][tok, :]   M=128 rows, N=64 tokens, K=576
// itself, so the pair exchanges nothing: both CTAs hold the same scores and
// take the same decisions (the same instructions on the same bits). The
// queries (128 x 576 x 2 B = 147 KB) do not fit in shared memory beside the
// full-width tiles, so latent columns 0-255 of Q sit in tensor memory and are
// the score product's A operand there (as P is the PV product's), and latent
// columns 256-511 with the 64 rope columns stay in shared memory.
//
// TMEM: O 256 columns, S 2 x 64 (the probabilities overwrite the scores in
// place, hi and lo terms for bf16), Q 128 (256 columns packed two per
// column) = 512. Shared memory: Q (4 swizzled [128 x 64] chunks and two
// [128 x 32] rope boxes with the 64-byte swizzle, 80 KB) and two full-width
// 64-token tile slots of 72 KB (both halves of ckv as one 4D TMA box per page
// each, and both 32-column kpe boxes): 227 KB with the barriers. A slot is
// two parts with barriers of their own: this CTA's ckv half (the V operand,
// free once PV is done) and the other half with the kpe (read by the score
// product only, free once it is done), so the next tile's larger part loads
// while PV still runs.
//
// Warp roles (384 threads): warps 0-7 softmax and epilogue (thread = row r =
// TMEM lane 32 (w % 4) + lane; warps w and w + 4 share the rows and take the
// two 32-token halves of each tile), warp 8 TMEM owner + MMA issuer, warps
// 9-11 page producers.
#include "device_common.cuh"

namespace mla {

namespace {

constexpr int kT = 64;                            // tokens per tile
constexpr int kRows = 128;                        // query rows (M)
constexpr int kHalfBoxes = 4;                     // ckv column blocks per half: 256 columns
constexpr int kHalfCols = kHalfBoxes * kBoxCols;  // 256
constexpr int kGroupBytes = 8 * kHalfCols * 2;    // 4 KB: one 8-token group of a half's four blocks
constexpr int kCkvBytes = kT * kHalfCols * 2;     // 32 KB: one half of a tile's ckv
constexpr int kKpeCols = kRope / 2;               // 32 rope columns a box
constexpr int kKpeBytes = kT * kKpeCols * 2;      // 4 KB: [64 tokens x 32 columns], 64-byte swizzle
constexpr int kTileSlot = 2 * kCkvBytes + 2 * kKpeBytes;  // 72 KB
constexpr int kSlots = 2;
constexpr int kPrefetch = 3;                      // tiles ahead of the one being loaded that are prefetched to L2
constexpr int kQChunk = kRows * 128;              // 16 KB: [128 rows x 64 columns], swizzled
constexpr int kQKpe = kRows * kKpeCols * 2;       // 8 KB: [128 rows x 32 rope columns], 64-byte swizzle
constexpr int kPageWarps = 3;
constexpr int kSoftmaxWarps = 8;
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kMmaWarp = kSoftmaxWarps;
constexpr int kThreads = (kSoftmaxWarps + 1 + kPageWarps) * 32;  // 384
constexpr int kHalfT = kT / 2;
constexpr float kRescaleTau = 8.0f;

constexpr uint32_t kOffQ = 0;                              // 64 KB: latent columns 256-511
constexpr uint32_t kOffQKpe = 4 * kQChunk;                 // 16 KB: the two rope boxes
constexpr uint32_t kOffTile = kOffQKpe + 2 * kQKpe;        // 80 KB: 2 tile slots
constexpr uint32_t kOffSmall = kOffTile + kSlots * kTileSlot;  // 224 KB
constexpr uint32_t kSmem = kOffSmall + 2048 + 1024;        // + alignment slack
static_assert(kTileSlot % 1024 == 0 && kOffTile % 1024 == 0, "swizzle atoms stay aligned");
static_assert(kSmem <= 232448, "shared memory per CTA");

constexpr uint32_t kTmemO = 0;      // O [128 x 256] fp32
constexpr uint32_t kTmemS = 256;    // S [128 x 64] fp32, then P in place; 2 buffers
constexpr uint32_t kTmemQ = 384;    // Q latent columns 0-255, 16-bit, two a column
constexpr uint32_t kTmemCols = 512;

struct Small {
  // a slot in two parts: this CTA's ckv half (the V operand, free once PV is done) and the other ckv half
  // with both kpe boxes (read by the score product only, free once it is done)
  uint64_t full[kSlots], empty[kSlots], fullb[kSlots], emptyb[kSlots], sfull[2], ppfull[2], pvdone[2], drain;
  uint32_t tmem_base;
  int32_t abort_flag;
  float half_val[2][kRows];  // per row, the two token halves' tile maximum (then their sums)
};
static_assert(sizeof(Small) <= 2048, "small smem region");

__device__ __forceinline__ uint32_t tmem_lane_base(int warp) { return static_cast<uint32_t>(32 * (warp & 3)) << 16; }

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (BF16) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
  } else {
    const __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
}
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    mla_partial_mh_nx_kernel(const __grid_constant__ CUtensorMap tm_pages,
                             const __grid_constant__ CUtensorMap tm_kpe_half, const PartialParams p) {
  extern __shared__ uint8_t smem_raw[];
  pdl_launch_dependents();  // the merge of these partials may be scheduled now; it waits for this grid
  uint8_t* smem = align1024(smem_raw);
  uint8_t* qs = smem + kOffQ;
  Small* sm = reinterpret_cast<Small*>(smem + kOffSmall);
  volatile int32_t* abort_flag = &sm->abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int half = static_cast<int>(cluster_ctarank() & 1u);
  const int rows_total = p.q_len * p.H;

  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&sm->full[s], kPageWarps);  // one expect_tx arrival per producer warp
      mbar_init(&sm->empty[s], 1);
      mbar_init(&sm->fullb[s], kPageWarps);
      mbar_init(&sm->emptyb[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm->sfull[t], 1);
      mbar_init(&sm->ppfull[t], kSoftmaxWarps);
      mbar_init(&sm->pvdone[t], 1);
    }
    mbar_init(&sm->drain, 1);
    sm->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&sm->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  // both CTAs of the pair take the whole chunk; pair g = blockIdx.x / 2 takes query rows [128 g, 128 g + 128)
  const CtaWork w = cta_work(p, kRows, kT, 0, 1, -1, static_cast<int32_t>(blockIdx.x >> 1));
  const int ntiles = (w.sub1 - w.sub0 + kT - 1) / kT;

  if (warp > kMmaWarp) {
    // ------------------------------------------------------------------ producers
    const int k0 = warp - kMmaWarp - 1;  // this warp loads pages k0, k0 + 3, ... of each tile (at most 2)
    const uint64_t pol = l2_policy_evict_first();
    uint64_t tmo = p.timeout_ns;
    asm volatile("" : "+l"(tmo));
    const int npages_req = (w.L + p.bs - 1) / p.bs;
    int win_base = -1, win_pid = -1;
    auto page_of = [&](int pg) -> int {  // warp-uniform pg
      const int base = pg & ~31;
      if (base != win_base) {
        win_base = base;
        const int q = base + lane;
        win_pid = (q < npages_req && q < p.max_blocks) ? checked_page(p, w.b, q) : -1;
      }
      return __shfl_sync(0xffffffffu, win_pid, pg & 31);
    };
    int issued_b = -1, issued_a = -1;  // the last tile whose score-only part, V half this warp issued
    for (int i = 0; i < ntiles; ++i) {
      const int s = i % kSlots;
      const int tok0 = w.sub0 + i * kT;
      const int pg0 = tok0 / p.bs;
      const int npg = (min(kT, w.sub1 - tok0) + p.bs - 1) / p.bs;
      const int mine = (npg > k0) ? (npg - k0 + kPageWarps - 1) / kPageWarps : 0;  // at most 2 (bs >= 16)
      int pids[2];
#pragma unroll
      for (int m = 0; m < 2; ++m) pids[m] = (m < mine) ? page_of(pg0 + k0 + m * kPageWarps) : -1;
      uint8_t* slot = smem + kOffTile + s * kTileSlot;
      const int other = half ^ 1;
      // the score-only part first (the other ckv half, both kpe boxes): free once S(i-2) is done
      if (i >= kSlots) {
        int ok = 1;
        if (lane == 0) {
          ok = mbar_wait(&sm->emptyb[s], ((i / kSlots) - 1) & 1, tmo) && !*abort_flag;
          if (!ok) *abort_flag = 1;
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
      if (lane == 0)
        mbar_arrive_expect_tx(&sm->fullb[s], static_cast<uint32_t>(mine * p.bs * (kHalfCols + 2 * kKpeCols) * 2));
      __syncwarp();
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        if (lane == m && m < mine) {
          const int j = k0 + m * kPageWarps;
          tma_load_4d(slot + other * kCkvBytes + j * p.bs * (kHalfCols * 2), &tm_pages, 0, 0, kHalfBoxes * other,
                      pids[m] * (p.bs / 8), &sm->fullb[s], pol);
#pragma unroll
          for (int h = 0; h < 2; ++h)
            tma_load_2d(slot + 2 * kCkvBytes + h * kKpeBytes + j * p.bs * (kKpeCols * 2), &tm_kpe_half, kKpeCols * h,
                        pids[m] * p.bs, &sm->fullb[s], pol);
        }
      }
      issued_b = i;
      // then this CTA's ckv half (the V operand): free once PV(i-2) is done
      if (i >= kSlots) {
        int ok = 1;
        if (lane == 0) {
          ok = mbar_wait(&sm->empty[s], ((i / kSlots) - 1) & 1, tmo) && !*abort_flag;
          if (!ok) *abort_flag = 1;
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
      if (lane == 0) mbar_arrive_expect_tx(&sm->full[s], static_cast<uint32_t>(mine * p.bs * kHalfCols * 2));
      __syncwarp();
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        if (lane == m && m < mine) {
          const int j = k0 + m * kPageWarps;
          tma_load_4d(slot + half * kCkvBytes + j * p.bs * (kHalfCols * 2), &tm_pages, 0, 0, kHalfBoxes * half,
                      pids[m] * (p.bs / 8), &sm->full[s], pol);
        }
      }
      issued_a = i;
      // an L2 prefetch of tile i + kPrefetch's pages (latent rows by the even CTA, rope rows by the odd one),
      // so that its slot load, which waits for PV(i + kPrefetch - 2) to free the slot, reads L2
      if (i + kPrefetch < ntiles) {
        const int qtok0 = w.sub0 + (i + kPrefetch) * kT;
        const int qg0 = qtok0 / p.bs;
        const int qn = (min(kT, w.sub1 - qtok0) + p.bs - 1) / p.bs;
        for (int j = k0; j < qn; j += kPageWarps) {
          const int qpid = page_of(qg0 + j);
          if (lane == 0 && qpid >= 0) {
            const long long row = static_cast<long long>(qpid) * p.bs;
            if (half == 0)
              bulk_prefetch_l2(p.ckv + row * (kRank * 2), static_cast<uint32_t>(p.bs * kRank * 2));
            else
              bulk_prefetch_l2(p.kpe + row * (kRope * 2), static_cast<uint32_t>(p.bs * kRope * 2));
          }
        }
      }
    }
    // after an abort, let this warp's loads still in flight land before shared memory is released
    if (lane == 0 && *abort_flag) {
      for (int t = max(0, issued_b - (kSlots - 1)); t <= issued_b; ++t)
        mbar_wait(&sm->fullb[t % kSlots], (t / kSlots) & 1, kDrainTimeoutNs);
      for (int t = max(0, issued_a - (kSlots - 1)); t <= issued_a; ++t)
        mbar_wait(&sm->full[t % kSlots], (t / kSlots) & 1, kDrainTimeoutNs);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    const uint32_t idesc_s = idesc_f16_f32(kRows, kT, BF16, false, false);         // A = Q, B = K tile
    const uint32_t idesc_o = idesc_f16_f32(kRows, kHalfCols, BF16, false, true);   // A = P (TMEM), B = V N-major
    const uint32_t q_base = smem_u32(qs);
    const uint32_t tile_base = smem_u32(smem + kOffTile);
    uint64_t tmo = p.timeout_ns;
    asm volatile("" : "+l"(tmo));
    // score product of tile i into S buffer i & 1, K = 576 in order: latent columns 0-255 (Q from tensor
    // memory, the tile's first half), 256-511 (Q from shared memory, the second half), then the rope
    // columns (two 64-byte-swizzled boxes of two K steps each)
    auto score = [&](int i) {
      const int t = i & 1;
      if (lane == 0) {
        tc_fence_after();
        const uint32_t slot = tile_base + (i % kSlots) * kTileSlot;
        const uint32_t d = tmem + kTmemS + t * kT;
#pragma unroll
        for (int c = 0; c < kHalfBoxes; ++c) {
          const uint64_t kd = smem_desc_sw128(slot + c * 1024, 16, kGroupBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_f16_ts(d, tmem + kTmemQ + 8 * (4 * c + kk), desc_add(kd, kk * 32), idesc_s,
                        (c == 0 && kk == 0) ? 0u : 1u);
        }
#pragma unroll
        for (int c = 0; c < kHalfBoxes; ++c) {
          const uint64_t qd = smem_desc_sw128(q_base + c * kQChunk, 16, 1024);
          const uint64_t kd = smem_desc_sw128(slot + kCkvBytes + c * 1024, 16, kGroupBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) umma_f16_ss(d, desc_add(qd, kk * 32), desc_add(kd, kk * 32), idesc_s, 1u);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint64_t qd = smem_desc_sw64(q_base + kOffQKpe + h * kQKpe, 512);
          const uint64_t kd = smem_desc_sw64(slot + 2 * kCkvBytes + h * kKpeBytes, 512);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) umma_f16_ss(d, desc_add(qd, kk * 32), desc_add(kd, kk * 32), idesc_s, 1u);
        }
        umma_commit(&sm->sfull[t]);
        umma_commit(&sm->emptyb[i % kSlots]);  // the score-only part of the slot is free
      }
      __syncwarp();
    };
    // rows [nvalid, nend) of this CTA's ckv half of a slot: zeroed so the V operand stays finite
    auto zero_rows = [&](uint8_t* ckv, int nvalid, int nend) {
      for (int x = lane; x < (nend - nvalid) * kHalfBoxes * 8; x += 32) {
        const int rc = x >> 3, tok = nvalid + rc / kHalfBoxes, c = rc % kHalfBoxes;
        *reinterpret_cast<uint4*>(ckv + (tok >> 3) * kGroupBytes + c * 1024 + (tok & 7) * 128 + (x & 7) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
    };
    auto pv = [&](int i) {
      const int t = i & 1, s = i % kSlots;
      const int nvalid = min(kT, w.sub1 - (w.sub0 + i * kT));
      const int ksteps = (nvalid + 15) >> 4;
      if (nvalid < (ksteps << 4)) {
        zero_rows(smem + kOffTile + s * kTileSlot + half * kCkvBytes, nvalid, ksteps << 4);
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        tc_fence_after();
        const uint32_t v_half = tile_base + s * kTileSlot + half * kCkvBytes;
        const uint32_t pa = tmem + kTmemS + t * kT;
        for (int ks = 0; ks < ksteps; ++ks) {
          const uint64_t vd = smem_desc_sw128(v_half + ks * 2 * kGroupBytes, 1024, kGroupBytes);
          // K step ks: tokens [16 ks, 16 ks + 16) of token half ks / 2, whose P (hi, then lo) fills
          // the first 16 (then the next 16) of that half's 32 columns of the buffer
          const uint32_t pk = pa + 32 * (ks >> 1) + 8 * (ks & 1);
          umma_f16_ts(tmem + kTmemO, pk, vd, idesc_o, (i > 0 || ks > 0) ? 1u : 0u);
          if (BF16) umma_f16_ts(tmem + kTmemO, pk + 16, vd, idesc_o, 1u);
        }
        umma_commit(&sm->empty[s]);
        umma_commit(&sm->pvdone[t]);
      }
      __syncwarp();
    };
    named_bar_sync(2, kSoftmaxThreads + 32);  // Q staged by the softmax warps (shared and tensor memory)
    // Issue as the inputs get ready, each product in tile order: PV(np) once its probabilities are in
    // TMEM, else S(ns) once tile ns has landed and its buffer is free (PV(ns-2) done). Nothing ready for
    // longer than the wait limit (or an abort elsewhere) ends it.
    int ns = 0, np = 0;
    bool idle = false;
    uint64_t idle_t0 = 0;
    while (np < ntiles) {
      int act = 0;
      if (lane == 0) {
        if (np < ns && mbar_test(&sm->ppfull[np & 1], (np >> 1) & 1)) {
          act = 2;
        } else if (ns < ntiles && (ns < 2 || mbar_test(&sm->pvdone[ns & 1], ((ns >> 1) - 1) & 1)) &&
                   mbar_test(&sm->full[ns % kSlots], (ns / kSlots) & 1) &&
                   mbar_test(&sm->fullb[ns % kSlots], (ns / kSlots) & 1)) {
          act = 1;
        } else if (*abort_flag) {
          act = -1;
        } else {
          const uint64_t now = globaltimer_ns();
          if (!idle) {
            idle = true;
            idle_t0 = now;
          } else if (now - idle_t0 > tmo) {
            act = -1;
            *abort_flag = 1;
            flag_error(MLA_DEVERR_TIMEOUT);
          }
        }
        if (act > 0) idle = false;
      }
      act = __shfl_sync(0xffffffffu, act, 0);
      if (act == 2) {
        pv(np);
        ++np;
      } else if (act == 1) {
        score(ns);
        ++ns;
      } else if (act < 0) {
        break;
      }
    }
    if (lane == 0) {  // every MMA issued so far has completed before TMEM is read or freed
      umma_commit(&sm->drain);
      mbar_wait(&sm->drain, 0, kDrainTimeoutNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax: thread = row
    const int r = 32 * (warp & 3) + lane;  // query row of this thread (TMEM lane r)
    const int hf = warp >> 2;               // its token half of each tile: tokens [32 hf, 32 hf + 32)
    const uint32_t lane_base = tmem_lane_base(warp);
    const bool real = r < w.nrows;
    const long long qrow = static_cast<long long>(w.b) * rows_total + w.row0 + (real ? r : 0);
    // Q latent columns 256-511 (4 chunks, 128-byte swizzle) and the 64 rope columns (two boxes, 64-byte
    // swizzle) into shared memory, K-major, all the 16-byte copies in flight at once; rows past the
    // group's zero-filled
    constexpr int kQPieces = (kHalfCols + kRope) / 8;  // 16-byte pieces per row: 40
    for (int idx = tid; idx < kRows * kQPieces; idx += kSoftmaxThreads) {
      const int rr = idx / kQPieces, k = (idx % kQPieces) * 8;
      const bool in = rr < w.nrows;
      const long long row = static_cast<long long>(w.b) * rows_total + w.row0 + (in ? rr : 0);
      const uint16_t* src = (k < kHalfCols) ? p.q_abs + row * kRank + kHalfCols + k : p.q_pe + row * kRope + (k - kHalfCols);
      const int kr = k - kHalfCols;
      uint8_t* dst = (k < kHalfCols) ? qs + (k / kBoxCols) * kQChunk + sw128_offset(rr, k % kBoxCols)
                                     : qs + kOffQKpe + (kr / kKpeCols) * kQKpe + sw64_offset(rr, kr % kKpeCols);
      cp_async16(dst, src, in ? 16u : 0u);
    }
    // Q latent columns [128 hf, 128 hf + 128) of this thread's row into tensor memory, two 16-bit values a
    // column (element 2u in the low half, as they lie in memory)
    {
      const uint4* src = reinterpret_cast<const uint4*>(p.q_abs + qrow * kRank + 128 * hf);
#pragma unroll
      for (int g = 0; g < 4; ++g) {  // 32 values = 16 columns a step
        float v[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 x = real ? src[4 * g + u] : make_uint4(0u, 0u, 0u, 0u);
          v[4 * u] = __uint_as_float(x.x);
          v[4 * u + 1] = __uint_as_float(x.y);
          v[4 * u + 2] = __uint_as_float(x.z);
          v[4 * u + 3] = __uint_as_float(x.w);
        }
        tmem_st16(tmem + lane_base + kTmemQ + 64 * hf + 16 * g, v);
      }
      tmem_wait_st();
    }
    cp_async_wait_all();
    fence_proxy_async_smem();
    tc_fence_before();
    named_bar_arrive(2, kSoftmaxThreads + 32);

    float scale_log2 = p.scale_log2;
    uint64_t tmo = p.timeout_ns;
    asm volatile("" : "+f"(scale_log2), "+l"(tmo));
    // visible tokens of this row: t < L, and t <= L - q_len + i under the causal rule
    const int row_q = (w.row0 + r) / p.H;
    const int tlim = min(w.sub1, p.causal ? (w.L - p.q_len + row_q + 1) : w.L);
    float m_r = -INFINITY, l_r = 0.f;
    for (int i = 0; i < ntiles; ++i) {
      const int buf = i & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&sm->sfull[buf], (i >> 1) & 1, tmo);
      ok = __all_sync(0xffffffffu, __shfl_sync(0xffffffffu, ok, 0));
      float x[kHalfT];
      float mx = -INFINITY;
      const uint32_t sa = tmem + lane_base + kTmemS + buf * kT + 32 * hf;
      if (ok) {
        tc_fence_after();
        tmem_ld16(sa, x);
        tmem_ld16(sa + 16, x + 16);
        tmem_wait_ld();
        const int nvis = min(kT, tlim - (w.sub0 + i * kT)) - kHalfT * hf;  // tokens of this half the row sees
        if (__builtin_expect(nvis < kHalfT, 0)) {
#pragma unroll
          for (int t = 0; t < kHalfT; ++t) x[t] = (t < nvis) ? x[t] * scale_log2 : -INFINITY;
        } else {
#pragma unroll
          for (int t = 0; t < kHalfT; ++t) x[t] *= scale_log2;
        }
#pragma unroll
        for (int t = 0; t < kHalfT; ++t) mx = fmaxf(mx, x[t]);
      }
      sm->half_val[hf][r] = mx;
      if (named_bar_sync_or(1, kSoftmaxThreads, !ok || *abort_flag != 0)) {
        if (lane == 0) *abort_flag = 1;
        break;
      }
      mx = fmaxf(mx, sm->half_val[hf ^ 1][r]);  // the row's maximum over the tile: the same in both halves
      named_bar_sync(3, kSoftmaxThreads);        // both halves have read it before either writes the next
      // lazy rescale of this row (rare): move the reference max and scale O and the sum; PV(i-1) must be
      // complete before O is rescaled
      const bool need = mx > m_r + kRescaleTau;
      if (__builtin_expect(__any_sync(0xffffffffu, need), 0)) {
        const float m_new = need ? fmaxf(m_r, mx) : m_r;
        const float alpha = need ? ((m_r == -INFINITY) ? 0.f : exp2f(m_r - m_new)) : 1.f;
        if (i >= 1) {
          int ok2 = 1;
          if (lane == 0) ok2 = mbar_wait(&sm->pvdone[(i - 1) & 1], ((i - 1) >> 1) & 1, tmo);
          if (__shfl_sync(0xffffffffu, ok2, 0)) {
            tc_fence_after();
            for (int q = 0; q < kHalfCols / 32; ++q) {  // this thread's half of the row's O columns
              float v[16];
              const uint32_t a = tmem + lane_base + kTmemO + (kHalfCols / 2) * hf + q * 16;
              tmem_ld16(a, v);
              tmem_wait_ld();
#pragma unroll
              for (int jj = 0; jj < 16; ++jj) v[jj] *= alpha;
              tmem_st16(a, v);
            }
            tmem_wait_st();
          } else if (lane == 0) {
            *abort_flag = 1;
          }
        }
        l_r *= alpha;
        m_r = m_new;
      }
      // probabilities of tile i over this thread's 32 tokens -> the same 32 columns (hi, then lo)
      const float m_sub = (m_r == -INFINITY) ? 0.f : m_r;  // a row with no visible token yet: a finite stand-in
      float hw[16], lw[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const float p0 = fast_exp2(x[2 * u] - m_sub);  // masked scores (-inf) give 0
        const float p1 = fast_exp2(x[2 * u + 1] - m_sub);
        const uint32_t hpk = pack2<BF16>(p0, p1);
        hw[u] = __uint_as_float(hpk);
        const float h0 = h2f<BF16>(static_cast<uint16_t>(hpk & 0xffffu));
        const float h1 = h2f<BF16>(static_cast<uint16_t>(hpk >> 16));
        if (BF16) {
          const uint32_t lpk = pack2<BF16>(p0 - h0, p1 - h1);
          lw[u] = __uint_as_float(lpk);
          l_r += (h0 + h2f<BF16>(static_cast<uint16_t>(lpk & 0xffffu))) + (h1 + h2f<BF16>(static_cast<uint16_t>(lpk >> 16)));
        } else {
          lw[u] = 0.f;
          l_r += h0 + h1;
        }
      }
      tmem_st16(sa, hw);
      if (BF16) tmem_st16(sa + 16, lw);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->ppfull[buf]);
    }
    const bool aborted = named_bar_sync_or(1, kSoftmaxThreads, *abort_flag != 0);
    if (ntiles > 0 && !aborted) {
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&sm->pvdone[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, tmo);
      if (!__shfl_sync(0xffffffffu, ok, 0) && lane == 0) *abort_flag = 1;
    }
    sm->half_val[hf][r] = l_r;
    const bool read_o = (ntiles > 0) && !named_bar_sync_or(1, kSoftmaxThreads, *abort_flag != 0);  // uniform
    const float l_row = sm->half_val[0][r] + sm->half_val[1][r];  // the row's sum, the same in both halves
    // epilogue: the normalized partial of this row over this thread's half of the CTA's 256 columns,
    // and the LSE (rank 0)
    const bool has_mass = read_o && real && (m_r != -INFINITY) && (l_row > 0.f);
    const float inv = has_mass ? 1.f / l_row : 0.f;
    const long long orow = static_cast<long long>(w.slot) * rows_total + w.row0 + r;
    if (read_o) tc_fence_after();
    for (int q = 0; q < kHalfCols / 32; ++q) {
      float v[16];
      const int col = (kHalfCols / 2) * hf + q * 16;
      if (read_o) {
        tmem_ld16(tmem + lane_base + kTmemO + col, v);
        tmem_wait_ld();
      }
      if (real) {
        float4* dst = reinterpret_cast<float4*>(p.partials + orow * kRank + kHalfCols * half + col);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          dst[j] = has_mass ? make_float4(v[4 * j] * inv, v[4 * j + 1] * inv, v[4 * j + 2] * inv, v[4 * j + 3] * inv)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    if (half == 0 && hf == 0 && real) p.lse[orow] = has_mass ? m_r + log2f(l_row) : -INFINITY;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool BF16>
cudaError_t prepare_nx() {
  static bool done = false;
  if (done) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&mla_partial_mh_nx_kernel<BF16>),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e == cudaSuccess) done = true;
  return e;
}

}  // namespace

cudaError_t launch_partial_mh_nx(const CUtensorMap& tm_pages, const CUtensorMap& tm_kpe_half, const PartialParams& p,
                                 int num_chunks, bool bf16, cudaStream_t stream) {
  if (p.fp8) return cudaErrorInvalidValue;  // 16-bit caches only
  const cudaError_t e = bf16 ? prepare_nx<true>() : prepare_nx<false>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * ((p.q_len * p.H + kRows - 1) / kRows), num_chunks, 1);  // one CTA pair per 128-row group
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return bf16 ? cudaLaunchKernelEx(&cfg, mla_partial_mh_nx_kernel<true>, tm_pages, tm_kpe_half, p)
              : cudaLaunchKernelEx(&cfg, mla_partial_mh_nx_kernel<false>, tm_pages, tm_kpe_half, p);
}

cudaError_t mh_nx_read_clear_error(uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_device_error, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(uint32_t));
}

}  // namespace mla
