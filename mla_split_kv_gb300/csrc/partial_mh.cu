// Tensor-core partial-decode kernel for groups of 128 query rows (the heads of
// a many-head decode, e.g. H=128 with one query token, or the rows of a
// verify window, q_len x H), each group on a pair of CTAs, sm_103a.
//
// The operation is the one of the other partial kernels ("feat(core):
// matrix-absorbed MLA decode over a compressed-latent KV cache", *What
// changed*: SDPA(q_absorbed, ckv, ckv, scale, mask = scale * q_pe @ kpe^T),
// each chunk yielding a normalized partial and its log2 LSE).
//
// With 128 rows sharing each latent tile the two products are dense enough to
// keep the rows on the MMA's M side:
//   S[row, tok]  = Q[row, :] . [ckv | kpe][tok, :]        M=128 rows, N=64 tokens
//   O[row, d]   += P[row, tok] . ckv[tok, d]              M=128 rows, N=256 columns, K=64
// O for 128 rows x 512 columns would fill all of tensor memory, so the two
// CTAs of a cluster pair split the latent columns: CTA `half` holds ckv
// columns [256 half, 256 half + 256) (and the kpe box, of whose 4 16-column
// K steps it uses 2) and accumulates O for those columns. Each computes S
// over its columns (128 x 64 fp32), sends it from registers into the peer's
// shared memory with asynchronous 16-byte remote stores completing on the
// peer's mbarrier (no staging copy in its own shared memory), and adds the
// peer's part in a fixed order, so both hold the same scores and take the
// same decisions.
//
// S lands in TMEM with row r in lane r, so softmax thread r owns row r: its
// running max and sum are thread-local (no cross-thread reduction). It writes
// the probabilities back into TMEM in the same lane, packed two 16-bit values
// per column, where the PV MMA reads them as its A operand; V (B operand) is
// the same shared-memory tile read N-major. With bf16 inputs P is carried as
// two bf16 terms (hi + lo, two MMAs per step), as in the other kernels.
//
// TMEM: O 256 columns, S 2 x 64, P 2 x (32 + 32) = 512. Shared memory: Q (4
// swizzled [128 x 64] chunks of this CTA's latent columns and its 32 rope
// columns with the 64-byte swizzle, 72 KB), three 64-token tile slots of 36 KB
// (the ckv half as one 4D TMA box per page: row groups of four [8 x 64] atoms,
// group g and block c at 4096 g + 1024 c; this CTA's 32 kpe columns, 64-byte
// swizzle), so tiles i+1 and i+2 load while tile i is computed, and the peer's
// partial S (32 KB): 215 KB.
//
// Warp roles (384 threads): warps 0-7 softmax and epilogue (thread = row r =
// TMEM lane 32 (w % 4) + lane; warps w and w + 4 share the rows and take the
// two 32-token halves of each tile, which halves each thread's exponentials
// and conversions and puts two softmax warps on every scheduler), warp 8 TMEM
// owner + MMA issuer, warps 9-11 page producers.
#include "device_common.cuh"

namespace mla {

namespace {

constexpr int kT = 64;                            // tokens per tile
constexpr int kRows = 128;                        // query rows (M)
constexpr int kHalfBoxes = 4;                     // ckv column blocks per CTA: 256 columns
constexpr int kHalfCols = kHalfBoxes * kBoxCols;  // 256
constexpr int kGroupBytes = 8 * kHalfCols * 2;    // 4 KB: one 8-token group of the four blocks
constexpr int kCkvBytes = kT * kHalfCols * 2;     // 32 KB
constexpr int kKpeCols = kRope / 2;               // 32 rope columns per CTA
constexpr int kKpeBytes = kT * kKpeCols * 2;      // 4 KB: [64 tokens x 32 columns], 64-byte swizzle
constexpr int kTileSlot = kCkvBytes + kKpeBytes;  // 36 KB
constexpr int kSlots = 3;
constexpr int kQChunk = kRows * 128;              // 16 KB: [128 rows x 64 columns], swizzled
constexpr int kQKpe = kRows * kKpeCols * 2;       // 8 KB: [128 rows x 32 rope columns], 64-byte swizzle
constexpr int kPageWarps = 3;
constexpr int kSoftmaxWarps = 8;                  // two per TMEM lane quadrant: each takes half of a tile's tokens
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kMmaWarp = kSoftmaxWarps;
constexpr int kThreads = (kSoftmaxWarps + 1 + kPageWarps) * 32;  // 384: three warps per scheduler
constexpr int kHalfT = kT / 2;                    // tokens of a tile per softmax thread
constexpr float kRescaleTau = 8.0f;

constexpr uint32_t kOffQ = 0;                             // 64 KB: latent columns
constexpr uint32_t kOffQKpe = 4 * kQChunk;                // 8 KB: rope columns
constexpr uint32_t kOffTile = kOffQKpe + kQKpe;           // 72 KB: 3 tile slots
constexpr uint32_t kOffX = kOffTile + kSlots * kTileSlot; // 180 KB: the peer's partial S
constexpr uint32_t kXBytes = kRows * kT * 4;              // [128 rows][64 tokens] fp32: 32 KB
constexpr uint32_t kOffSmall = kOffX + kXBytes;           // 212 KB
constexpr uint32_t kSmem = kOffSmall + 2048 + 1024;       // + alignment slack
static_assert(kTileSlot % 1024 == 0 && kOffTile % 1024 == 0, "swizzle atoms stay aligned");
static_assert(kSmem <= 232448, "shared memory per CTA");

// E4M3 caches: a tile's bytes land unswizzled in the upper half of its slot (staged rows of 256 bytes:
// ckv tokens 0-63, then the kpe, 8 tokens a row) and are widened to fp16 in place
constexpr int kStage = kTileSlot - kT * (kHalfCols + kKpeCols);  // 18 KB
static_assert(kStage == 18432 && kCkvBytes == kStage + 56 * kHalfCols && kGroupBytes == 4096,
              "the widening order below assumes this geometry");

constexpr uint32_t kTmemO = 0;      // O [128 x 256] fp32
constexpr uint32_t kTmemS = 256;    // S [128 x 64] fp32, 2 buffers
constexpr uint32_t kTmemP = 384;    // P [128 x 64] 16-bit, hi and lo (32 columns each), 2 buffers
constexpr uint32_t kTmemCols = 512;

struct Small {
  uint64_t full[kSlots], empty[kSlots], sfull[2], sfree[2], ppfull[2], pvdone[2], xfull, xempty, drain;
  uint64_t landed[kSlots], conv;  // E4M3 caches: a tile's bytes landed; the producer warps' meeting point
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t peer_abort;        // set by the peer CTA (remote store) when it gave up
  float half_val[2][kRows];  // per row, the two token halves' tile maximum (then their sums)
};
static_assert(sizeof(Small) <= 2048, "small smem region");

__device__ __forceinline__ uint32_t tmem_lane_base(int warp) { return static_cast<uint32_t>(32 * (warp & 3)) << 16; }

// two values rounded to 16 bits in one conversion: a in the low half, b in the high half
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

// X16: the pair's partial scores cross as fp16 (an instance each, no run-time branch in the loop);
// FP8: E4M3 caches beside fp16 queries (BF16 false), widened in the tile slots, scaled on the output
template <bool BF16, bool X16, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
    mla_partial_mh_kernel(const __grid_constant__ CUtensorMap tm_pages, const __grid_constant__ CUtensorMap tm_kpe_half,
                          const PartialParams p) {
  extern __shared__ uint8_t smem_raw[];
  pdl_launch_dependents();  // the merge of these partials may be scheduled now; it waits for this grid
  uint8_t* smem = align1024(smem_raw);
  uint8_t* qs = smem + kOffQ;
  float* xs = reinterpret_cast<float*>(smem + kOffX);
  Small* sm = reinterpret_cast<Small*>(smem + kOffSmall);
  volatile int32_t* abort_flag = &sm->abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int half = static_cast<int>(rank & 1u);
  const int rows_total = p.q_len * p.H;

  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&sm->full[s], kPageWarps);  // one expect_tx arrival per producer warp
      mbar_init(&sm->empty[s], 1);
      mbar_init(&sm->landed[s], kPageWarps);
    }
    mbar_init(&sm->conv, kPageWarps);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm->sfull[t], 1);
      mbar_init(&sm->sfree[t], kSoftmaxWarps);
      mbar_init(&sm->ppfull[t], kSoftmaxWarps);
      mbar_init(&sm->pvdone[t], 1);
    }
    mbar_init(&sm->xfull, 1);   // local expect_tx arrival + the peer's st.async bytes
    mbar_init(&sm->xempty, kSoftmaxWarps);  // one remote arrival per peer softmax warp
    mbar_init(&sm->drain, 1);
    sm->abort_flag = 0;
    sm->peer_abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&sm->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive_release();  // the peer touches this CTA's barriers only after this cluster phase
  const uint32_t tmem = sm->tmem_base;
  // both CTAs of the pair take the whole chunk; pair g = blockIdx.x / 2 takes query rows [128 g, 128 g + 128)
  // (the row groups of a chunk are adjacent clusters, so they stream the same tiles at about the same time
  // and the later reads are served by L2)
  const CtaWork w = cta_work(p, kRows, kT, 0, 1, -1, static_cast<int32_t>(blockIdx.x >> 1));
  const int ntiles = (w.sub1 - w.sub0 + kT - 1) / kT;
  // only the group's real rows exchange their partial scores (a group of 64 rows, H=64, sends half),
  // 4 bytes a score, or 2 with the fp16 exchange; the peer's bytes of tile 0 may land before this
  // expectation: its arrival completes the phase
  constexpr bool x16 = X16;
  const uint32_t xbytes = static_cast<uint32_t>(min(w.nrows, kRows)) * kT * (x16 ? 2 : 4);
  if (tid == 0) mbar_arrive_expect_tx(&sm->xfull, xbytes);  // tile 0

  if (warp > kMmaWarp) {
    // ------------------------------------------------------------------ producers
    const int k0 = warp - kMmaWarp - 1;  // this warp loads pages k0, k0 + 3, ... of each tile (at most 2: 4 pages of 16)
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
    auto tile_pages = [&](int i, int* pg0, int* npg) {
      const int tok0 = w.sub0 + i * kT;
      *pg0 = tok0 / p.bs;
      *npg = (min(kT, w.sub1 - tok0) + p.bs - 1) / p.bs;
    };
    int issued = -1;  // the last tile whose loads this warp issued
    // the loads of this warp's pages of tile i into its slot (free), then (16-bit caches) an L2 prefetch
    // of the same pages of tile i+3: ckv by the even CTA, kpe by the odd one (with E4M3 caches the
    // prefetch measured slower: 388 against 355 us on the many-head decode)
    auto issue_tile = [&](int i) {
      const int s = i % kSlots;
      int pg0, npg;
      tile_pages(i, &pg0, &npg);
      const int mine = (npg > k0) ? (npg - k0 + kPageWarps - 1) / kPageWarps : 0;  // at most 2 (bs >= 16)
      int pids[2];
#pragma unroll
      for (int m = 0; m < 2; ++m) pids[m] = (m < mine) ? page_of(pg0 + k0 + m * kPageWarps) : -1;
      uint8_t* slot = smem + kOffTile + s * kTileSlot;
      constexpr int kElem = FP8 ? 1 : 2;  // bytes a cached value
      uint64_t* bar = FP8 ? &sm->landed[s] : &sm->full[s];
      if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(mine * p.bs * (kHalfCols + kKpeCols) * kElem));
      __syncwarp();
      // lane m issues this warp's page m (TMA issue from several lanes overlaps)
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        if (lane == m && m < mine) {
          const int j = k0 + m * kPageWarps;
          if constexpr (FP8) {  // bytes, unswizzled, into the upper part of the slot
            tma_load_2d(slot + kStage + j * p.bs * kHalfCols, &tm_pages, kHalfCols * half, pids[m] * p.bs, bar, pol);
            tma_load_2d(slot + kStage + kT * kHalfCols + j * p.bs * kKpeCols, &tm_kpe_half, kKpeCols * half,
                        pids[m] * p.bs, bar, pol);
          } else {
            tma_load_4d(slot + j * p.bs * (kHalfCols * 2), &tm_pages, 0, 0, kHalfBoxes * half, pids[m] * (p.bs / 8),
                        bar, pol);
            tma_load_2d(slot + kCkvBytes + j * p.bs * (kKpeCols * 2), &tm_kpe_half, kKpeCols * half, pids[m] * p.bs,
                        bar, pol);
          }
        }
      }
      issued = i;
      if (!FP8 && i + kSlots < ntiles) {
        int qg0, qn;
        tile_pages(i + kSlots, &qg0, &qn);
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
    };
    if constexpr (FP8) {
      // E4M3 caches: tile i's staged bytes become the 16-bit tile in place by the three producer warps,
      // a warp step taking two staged rows (512 bytes, 16 a lane). The 16-bit rows of ckv tokens 0-31 lie
      // below the staging; those of tokens 8g..8g+7 (g >= 4) overwrite staged rows 16g-72..16g-57 (from
      // row 0), and the 16-bit kpe staged rows 56-71. So, with the three warps meeting between the parts:
      // tokens 0-31 | tokens 32-47, then staged rows 48-71 into registers | those rows (tokens 48-63, the
      // kpe) from the registers. Lane 0 of each warp then counts it on the slot's full barrier. Lanes as
      // in the paired kernel: every quarter warp reads and writes 8 different 16-byte bank groups.
      const int r2 = (lane >> 2) & 1, cbl = (lane >> 3) ^ r2, kk = lane & 3;
      const int src_ckv = r2 * kHalfCols + cbl * 64 + kk * 16;
      const int tk_l = lane >> 1, hk = lane & 1;
      auto meet = [&](int phase) -> bool {  // two phases per tile; spins, the others being close
        __syncwarp();
        int ok = 1;
        if (lane == 0) {
          mbar_arrive(&sm->conv);
          if (!mbar_test(&sm->conv, phase & 1)) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_test(&sm->conv, phase & 1)) {
              if (globaltimer_ns() - t0 > tmo) {
                flag_error(MLA_DEVERR_TIMEOUT);
                ok = 0;
                break;
              }
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        __syncwarp();
        return ok != 0;
      };
      auto convert = [&](int i) -> bool {
        const int s = i % kSlots;
        const uint32_t slot = smem_u32(smem + kOffTile + s * kTileSlot);
        const uint32_t stage_src = slot + kStage + src_ckv;
        if (!__all_sync(0xffffffffu, mbar_wait(&sm->landed[s], (i / kSlots) & 1, tmo))) return false;
        widen_ckv_steps(slot, stage_src, 2 * k0, k0 == 0 ? 6 : 5, r2, cbl, kk);  // tokens 0-31: 16 steps
        if (!meet(2 * i)) return false;
        const int fb = (k0 + 2) % kPageWarps;  // rotated: 12 steps per warp over the tile
        widen_ckv_steps(slot, stage_src, 32 + 2 * fb, fb == 2 ? 2 : 3, r2, cbl, kk);  // tokens 32-47: 8 steps
        uint4 held[4];  // staged rows 48 + 2j, j = k0 + 3m: ckv tokens 48-63 (j < 8), then the kpe
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int j = k0 + kPageWarps * m;
          held[m] = lds128(slot + kStage + (48 + 2 * j) * kHalfCols + (j < 8 ? src_ckv : lane * 16));
        }
        if (!meet(2 * i + 1)) return false;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int j = k0 + kPageWarps * m;
          if (j < 8) {
            const int t = 48 + 2 * j, r = (t & 7) + r2;
            const uint32_t row = slot + (t >> 3) * kGroupBytes + cbl * 1024 + r * 128;
            widen16(held[m], row + (((2 * kk) ^ r) << 4), row + (((2 * kk + 1) ^ r) << 4));
          } else {  // kpe tokens 16 (j-8) .. +15: 32 bytes each, two 16-byte fp16 pieces per lane
            const int tk = 16 * (j - 8) + tk_l;
            const uint32_t row = slot + kCkvBytes + tk * (kKpeCols * 2);
            widen16(held[m], row + ((((2 * hk) ^ (tk >> 1)) & 3) << 4), row + ((((2 * hk + 1) ^ (tk >> 1)) & 3) << 4));
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->full[s]);
        return true;
      };
      // issue and widening interleave: the next tile's loads as soon as its slot is free, else the
      // widening of the oldest landed tile; nothing to do for longer than the wait limit (or an abort
      // elsewhere) ends it
      int ni = 0, nc = 0;
      bool idle = false;
      uint64_t idle_t0 = 0;
      while (nc < ntiles) {
        int act = 0;
        if (lane == 0) {
          if (ni < ntiles && ni < nc + kSlots &&
              (ni < kSlots || mbar_test(&sm->empty[ni % kSlots], ((ni / kSlots) - 1) & 1))) {
            act = 1;
          } else if (nc < ni && mbar_test(&sm->landed[nc % kSlots], (nc / kSlots) & 1)) {
            act = 2;
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
        if (act == 1) {
          issue_tile(ni++);
        } else if (act == 2) {
          if (!convert(nc)) {
            if (lane == 0) {
              *abort_flag = 1;
              flag_error(MLA_DEVERR_TIMEOUT);
            }
            break;
          }
          ++nc;
        } else if (act < 0) {
          break;
        }
      }
    } else {
      for (int i = 0; i < ntiles; ++i) {
        const int s = i % kSlots;
        if (i >= kSlots) {  // PV(i-3) released the slot
          int ok = 1;
          if (lane == 0) {
            ok = mbar_wait(&sm->empty[s], ((i / kSlots) - 1) & 1, tmo) && !*abort_flag;
            if (!ok) *abort_flag = 1;
          }
          if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        }
        issue_tile(i);
      }
    }
    // after an abort, let this warp's loads still in flight (the last three tiles it issued) land before
    // shared memory is released
    if (lane == 0 && *abort_flag)
      for (int t = max(0, issued - (kSlots - 1)); t <= issued; ++t)
        mbar_wait(FP8 ? &sm->landed[t % kSlots] : &sm->full[t % kSlots], (t / kSlots) & 1, kDrainTimeoutNs);
    cluster_wait_acquire();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    const uint32_t idesc_s = idesc_f16_f32(kRows, kT, BF16, false, false);         // A = Q, B = K tile
    const uint32_t idesc_o = idesc_f16_f32(kRows, kHalfCols, BF16, false, true);   // A = P (TMEM), B = V N-major
    const uint32_t q_base = smem_u32(qs);
    const uint32_t tile_base = smem_u32(smem + kOffTile);
    uint64_t tmo = p.timeout_ns;
    asm volatile("" : "+l"(tmo));
    // score product of tile i (slot i % 3) into S buffer i & 1: this CTA's 4 latent column blocks, then
    // its 32 rope columns (two K steps of the 64-byte-swizzled box)
    auto score = [&](int i) {
      const int t = i & 1;
      if (lane == 0) {
        tc_fence_after();
        const uint32_t slot = tile_base + (i % kSlots) * kTileSlot;
        const uint32_t d = tmem + kTmemS + t * kT;
#pragma unroll
        for (int c = 0; c < kHalfBoxes; ++c) {
          const uint64_t qd = smem_desc_sw128(q_base + c * kQChunk, 16, 1024);
          const uint64_t kd = smem_desc_sw128(slot + c * 1024, 16, kGroupBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_f16_ss(d, desc_add(qd, kk * 32), desc_add(kd, kk * 32), idesc_s, (c == 0 && kk == 0) ? 0u : 1u);
        }
        const uint64_t qd = smem_desc_sw64(q_base + kOffQKpe, 512);
        const uint64_t kd = smem_desc_sw64(slot + kCkvBytes, 512);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) umma_f16_ss(d, desc_add(qd, kk * 32), desc_add(kd, kk * 32), idesc_s, 1u);
        umma_commit(&sm->sfull[t]);
      }
      __syncwarp();
    };
    // rows [nvalid, nend) of the ckv part of a slot: zeroed so the V operand stays finite
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
        zero_rows(smem + kOffTile + s * kTileSlot, nvalid, ksteps << 4);
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        tc_fence_after();
        const uint32_t slot = tile_base + s * kTileSlot;
        const uint32_t pa = tmem + kTmemP + t * 64;
        for (int ks = 0; ks < ksteps; ++ks) {
          const uint64_t vd = smem_desc_sw128(slot + ks * 2 * kGroupBytes, 1024, kGroupBytes);
          // K step ks: tokens [16 ks, 16 ks + 16) of token half ks / 2, whose P (hi, then lo) fills
          // that half's 32 columns of the buffer
          const uint32_t pk = pa + 32 * (ks >> 1) + 8 * (ks & 1);
          umma_f16_ts(tmem + kTmemO, pk, vd, idesc_o, (i > 0 || ks > 0) ? 1u : 0u);
          if (BF16) umma_f16_ts(tmem + kTmemO, pk + 16, vd, idesc_o, 1u);
        }
        umma_commit(&sm->empty[s]);
        umma_commit(&sm->pvdone[t]);
      }
      __syncwarp();
    };
    named_bar_sync(2, kSoftmaxThreads + 32);  // Q staged by the softmax warps
    // Issue as the inputs get ready, each product in tile order: PV(np) once its probabilities are in
    // TMEM (first: it releases a slot for the next load), else S(ns) once tile ns has landed and its S
    // buffer is free. Nothing ready for longer than the wait limit (or an abort elsewhere) ends it.
    int ns = 0, np = 0;
    bool idle = false;
    uint64_t idle_t0 = 0;
    while (np < ntiles) {
      int act = 0;
      if (lane == 0) {
        if (np < ns && mbar_test(&sm->ppfull[np & 1], (np >> 1) & 1)) {
          act = 2;
        } else if (ns < ntiles && (ns < 2 || mbar_test(&sm->sfree[ns & 1], ((ns >> 1) - 1) & 1)) &&
                   mbar_test(&sm->full[ns % kSlots], (ns / kSlots) & 1)) {
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
    cluster_wait_acquire();
  } else {
    // ------------------------------------------------------------------ softmax (warps 0-3): thread = row
    // Q: this CTA's 256 latent columns (4 chunks, 128-byte swizzle), then its 32 rope columns (64-byte
    // swizzle); 128 rows, K-major (all the 16-byte copies in flight at once; rows past the request's
    // zero-filled)
    constexpr int kQPieces = (kHalfCols + kKpeCols) / 8;  // 16-byte pieces per row
    for (int idx = tid; idx < kRows * kQPieces; idx += kSoftmaxThreads) {
      const int r = idx / kQPieces, k = (idx % kQPieces) * 8;
      const bool in = r < w.nrows;
      const long long row = static_cast<long long>(w.b) * rows_total + w.row0 + (in ? r : 0);
      const uint16_t* src = (k < kHalfCols) ? p.q_abs + row * kRank + kHalfCols * half + k
                                            : p.q_pe + row * kRope + kKpeCols * half + (k - kHalfCols);
      uint8_t* dst = (k < kHalfCols) ? qs + (k / kBoxCols) * kQChunk + sw128_offset(r, k % kBoxCols)
                                     : qs + kOffQKpe + sw64_offset(r, k - kHalfCols);
      cp_async16(dst, src, in ? 16u : 0u);
    }
    cp_async_wait_all();
    fence_proxy_async_smem();
    named_bar_arrive(2, kSoftmaxThreads + 32);
    cluster_wait_acquire();  // the peer's barriers are initialised

    float scale_log2 = p.scale_log2;
    uint64_t tmo = p.timeout_ns;
    asm volatile("" : "+f"(scale_log2), "+l"(tmo));
    const int r = 32 * (warp & 3) + lane;  // query row of this thread (TMEM lane r)
    const int hf = warp >> 2;               // its token half of each tile: tokens [32 hf, 32 hf + 32)
    const uint32_t lane_base = tmem_lane_base(warp);
    // visible tokens of this row: t < L, and t <= L - q_len + i under the causal rule
    const int row_q = (w.row0 + r) / p.H;
    // end of the tokens this row sees in this CTA's range: the chunk end, and the causal limit
    const int tlim = min(w.sub1, p.causal ? (w.L - p.q_len + row_q + 1) : w.L);
    const uint32_t xsw = static_cast<uint32_t>(r & 15);
    const uint32_t peer_x = dsmem_addr(xs, peer);
    const uint32_t peer_xfull = dsmem_addr(&sm->xfull, peer);
    const uint32_t peer_xempty = dsmem_addr(&sm->xempty, peer);
    // row r of the receive buffer: 64 fp32 scores (16-byte chunk c at position c ^ (r & 15)), or with
    // the fp16 exchange 64 fp16 scores in the first half of the row's 256 bytes (c ^ (r & 7))
    const float4* xrow = reinterpret_cast<const float4*>(xs + r * kT);
    const uint32_t peer_xrow = peer_x + static_cast<uint32_t>(r * kT * 4);
    const uint32_t xsw8 = static_cast<uint32_t>(r & 7);
    float m_r = -INFINITY, l_r = 0.f;
    float own[kHalfT];  // this CTA's partial scores of the current tile, kept for B
    // C(j): probabilities of tile j (its scaled scores wait in its P buffer) -> the same buffer (hi, and lo
    // for bf16), 32 tokens at a time; then PV(j) may run
    auto probabilities = [&](int j) {
        // this thread's half of the buffer: its 32 scaled scores, overwritten by P hi (16 columns)
        // and, for bf16, P lo (16 columns)
        const uint32_t pa = tmem + lane_base + kTmemP + (j & 1) * 64 + 32 * hf;
        // a row that has seen no visible token yet has only -inf scores: subtract a finite stand-in
        const float m_sub = (m_r == -INFINITY) ? 0.f : m_r;
        float y[kHalfT];
        tc_fence_after();
        tmem_ld16(pa, y);
        tmem_ld16(pa + 16, y + 16);
        tmem_wait_ld();
        float hw[16], lw[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float p0 = fast_exp2(y[2 * u] - m_sub);  // masked scores (-inf) give 0
          const float p1 = fast_exp2(y[2 * u + 1] - m_sub);
          const uint32_t h = pack2<BF16>(p0, p1);  // one paired conversion, element 2u in the low half
          hw[u] = __uint_as_float(h);
          const float h0 = h2f<BF16>(static_cast<uint16_t>(h & 0xffffu));
          const float h1 = h2f<BF16>(static_cast<uint16_t>(h >> 16));
          if (BF16) {
            const uint32_t l = pack2<BF16>(p0 - h0, p1 - h1);
            lw[u] = __uint_as_float(l);
            l_r += (h0 + h2f<BF16>(static_cast<uint16_t>(l & 0xffffu))) + (h1 + h2f<BF16>(static_cast<uint16_t>(l >> 16)));
          } else {
            l_r += h0 + h1;
          }
        }
        tmem_st16(pa, hw);
        if (BF16) tmem_st16(pa + 16, lw);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->ppfull[j & 1]);
    };
    // Software pipeline over tiles: iteration i sends tile i's partial scores (A), computes the
    // probabilities of tile i-1 while those stores are in flight (C), then finishes tile i's scores (B).
    // Between B(i) and C(i) the scaled scores of tile i wait in tile i's P buffer in tensor memory
    // (64 fp32 columns), which C(i) then overwrites with the packed probabilities.
    for (int i = 0; i <= ntiles; ++i) {
      const bool cur = i < ntiles;
      const int buf = i & 1;
      int ok = 1;
      // C(i-1) is done while tile i's copy is in flight; but first, if tile i's scores are not ready
      // (the MMA warp may be waiting for PV(i-1), which needs C(i-1)), right away
      bool c_done = (i == 0);
      if (!c_done) {
        int ready = 0;
        if (cur && lane == 0) ready = mbar_test(&sm->sfull[buf], (i >> 1) & 1) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, ready, 0)) {
          probabilities(i - 1);
          c_done = true;
        }
      }
      // ---- A(i): this CTA's partial S of tile i -> the peer's shared memory (16-byte asynchronous
      // remote stores from registers, completing on the peer's xfull)
      if (cur) {
        if (lane == 0) ok = mbar_wait(&sm->sfull[buf], (i >> 1) & 1, tmo);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok) {
          tc_fence_after();
          tmem_ld16(tmem + lane_base + kTmemS + buf * kT + 32 * hf, own);
          tmem_ld16(tmem + lane_base + kTmemS + buf * kT + 32 * hf + 16, own + 16);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm->sfree[buf]);
          // the peer has read tile i-1's scores out of its buffer
          if (i >= 1) ok = mbar_wait_cluster(&sm->xempty, (i - 1) & 1, tmo);
        }
        ok = __all_sync(0xffffffffu, ok);
        if constexpr (X16) {  // both CTAs add the two parts rounded to fp16: the same values on both sides
#pragma unroll
          for (int t = 0; t < kHalfT; ++t) own[t] = h2f<false>(f2h<false>(own[t]));
        }
        if (ok && r < w.nrows) {
          if constexpr (X16) {
#pragma unroll
            for (int c = 0; c < kHalfT / 8; ++c) {
              float4 v;
              v.x = __uint_as_float(pack2<false>(own[8 * c], own[8 * c + 1]));
              v.y = __uint_as_float(pack2<false>(own[8 * c + 2], own[8 * c + 3]));
              v.z = __uint_as_float(pack2<false>(own[8 * c + 4], own[8 * c + 5]));
              v.w = __uint_as_float(pack2<false>(own[8 * c + 6], own[8 * c + 7]));
              dsmem_st_async_f32x4(peer_xrow + (((4 * hf + c) ^ xsw8) << 4), v, peer_xfull);
            }
          } else {
#pragma unroll
            for (int c = 0; c < kHalfT / 4; ++c)
              dsmem_st_async_f32x4(peer_xrow + (((8 * hf + c) ^ xsw) << 4),
                                   make_float4(own[4 * c], own[4 * c + 1], own[4 * c + 2], own[4 * c + 3]), peer_xfull);
          }
        }
      }
      // (no barrier here: each warp goes on to C(i-1) as soon as its own stores are issued; a failure
      // in A ends the loop at B's barrier, in every warp)
      const bool a_ok = ok != 0;
      // ---- C(i-1), when tile i's scores are not ready yet (so it cannot wait on them)
      if (!c_done) {
        probabilities(i - 1);
        c_done = true;
      }
      if (!cur) break;
      // ---- B(i): add the peer's part, scale and mask, lazy rescale, scores -> tile i's P buffer
      const int tok0 = w.sub0 + i * kT;
      ok = a_ok ? mbar_wait_cluster(&sm->xfull, i & 1, tmo) : 0;
      ok = __all_sync(0xffffffffu, ok);
      float x[kHalfT];
      float mx = -INFINITY;
      if (ok) {
#pragma unroll
        for (int c = 0; c < kHalfT / 4; ++c) {
          const float4 o = make_float4(own[4 * c], own[4 * c + 1], own[4 * c + 2], own[4 * c + 3]);
          // (a padding row past the group's rows takes no peer part: its scores are never used)
          float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
          if (r < w.nrows) {
            if constexpr (X16) {
              const uint4 q = reinterpret_cast<const uint4*>(xrow)[(4 * hf + (c >> 1)) ^ xsw8];
              const uint32_t a = (c & 1) ? q.z : q.x, b = (c & 1) ? q.w : q.y;
              y = make_float4(h2f<false>(static_cast<uint16_t>(a & 0xffffu)), h2f<false>(static_cast<uint16_t>(a >> 16)),
                              h2f<false>(static_cast<uint16_t>(b & 0xffffu)), h2f<false>(static_cast<uint16_t>(b >> 16)));
            } else {
              y = xrow[(8 * hf + c) ^ xsw];
            }
          }
          // rank-0 part + rank-1 part, the same sum in both CTAs
          x[4 * c] = half ? (y.x + o.x) : (o.x + y.x);
          x[4 * c + 1] = half ? (y.y + o.y) : (o.y + y.y);
          x[4 * c + 2] = half ? (y.z + o.z) : (o.z + y.z);
          x[4 * c + 3] = half ? (y.w + o.w) : (o.w + y.w);
        }
        __syncwarp();
        if (lane == 0) {
          // expect the peer's next tile before letting it send, then free the buffer (the values are
          // consumed above; a plain signal)
          if (tid == 0) mbar_arrive_expect_tx(&sm->xfull, xbytes);
          mbar_remote_arrive_relaxed(peer_xempty);
        }
        const int nvis = min(kT, tlim - tok0) - kHalfT * hf;  // tokens of this half the row can see
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
        *abort_flag = 1;
        break;
      }
      mx = fmaxf(mx, sm->half_val[hf ^ 1][r]);  // the row's maximum over the tile: the same in both halves
      // lazy rescale of this row (rare): move the reference max and scale O and the sum; PV(i-1)
      // (its probabilities were written in C(i-1) above) must be complete before O is rescaled
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
      // tile i's P buffer was last read by PV(i-2)
      if (i >= 2) {
        int ok3 = 1;
        if (lane == 0) ok3 = mbar_wait(&sm->pvdone[buf], ((i >> 1) - 1) & 1, tmo);
        if (!__shfl_sync(0xffffffffu, ok3, 0) && lane == 0) *abort_flag = 1;
      }
      {
        const uint32_t pa = tmem + lane_base + kTmemP + buf * 64 + 32 * hf;
        tmem_st16(pa, x);
        tmem_st16(pa + 16, x + 16);
        tmem_wait_st();
      }
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
    const bool has_mass = read_o && (r < w.nrows) && (m_r != -INFINITY) && (l_row > 0.f);
    // (an E4M3 cache's scale multiplies the output: folded into the normalisation)
    const float inv = has_mass ? (FP8 ? (1.f / l_row) * p.cache_scale : 1.f / l_row) : 0.f;
    const long long orow = static_cast<long long>(w.slot) * rows_total + w.row0 + r;
    if (read_o) tc_fence_after();
    for (int q = 0; q < kHalfCols / 32; ++q) {
      float v[16];
      const int col = (kHalfCols / 2) * hf + q * 16;
      if (read_o) {
        tmem_ld16(tmem + lane_base + kTmemO + col, v);
        tmem_wait_ld();
      }
      if (r < w.nrows) {
        float4* dst = reinterpret_cast<float4*>(p.partials + orow * kRank + kHalfCols * half + col);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          dst[j] = has_mass ? make_float4(v[4 * j] * inv, v[4 * j + 1] * inv, v[4 * j + 2] * inv, v[4 * j + 3] * inv)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    if (rank == 0 && hf == 0 && r < w.nrows) p.lse[orow] = has_mass ? m_r + log2f(l_row) : -INFINITY;
  }
  tc_fence_before();
  __syncthreads();
  // a CTA that gave up tells its peer before the last cluster barrier: the remote stores of partial
  // scores that either CTA issued may then still be in flight (writing the receiver's shared memory),
  // so after an abort on either side both stay until they have landed
  if (tid == 0 && *abort_flag) dsmem_st_u32(dsmem_addr(&sm->peer_abort, peer), 1u);
  cluster_sync();  // the peer is done with this CTA's shared memory
  if (*abort_flag || *reinterpret_cast<volatile int32_t*>(&sm->peer_abort)) settle_in_flight(20000ull);
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool BF16, bool X16, bool FP8>
cudaError_t prepare_mh() {
  static bool done = false;
  if (done) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&mla_partial_mh_kernel<BF16, X16, FP8>),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e == cudaSuccess) done = true;
  return e;
}

}  // namespace

// More than 16 rows (16 or fewer go to the paired 16-row kernel): groups of 128 rows, the last group
// padded (its rows past the end have zero queries and are not written back).
bool mh_supports(int total_rows, int cluster) { return total_rows > 16 && cluster == 2; }

cudaError_t launch_partial_mh(const CUtensorMap& tm_pages, const CUtensorMap& tm_kpe_half, const PartialParams& p,
                              int num_chunks, bool bf16, cudaStream_t stream) {
  const bool x16 = p.xchg16 != 0;
  if (p.fp8 && bf16) return cudaErrorInvalidValue;  // E4M3 caches go with fp16 queries
  cudaError_t e = p.fp8 ? (x16 ? prepare_mh<false, true, true>() : prepare_mh<false, false, true>())
                  : bf16 ? (x16 ? prepare_mh<true, true, false>() : prepare_mh<true, false, false>())
                         : (x16 ? prepare_mh<false, true, false>() : prepare_mh<false, false, false>());
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * ((p.q_len * p.H + kRows - 1) / kRows), num_chunks, 1);  // one CTA pair per 128-row group
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  // (not a programmatic dependent launch: with all SMs taken by one wave, launching early made the
  // many-head decode about 6 us per call slower)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.fp8)
    return x16 ? cudaLaunchKernelEx(&cfg, mla_partial_mh_kernel<false, true, true>, tm_pages, tm_kpe_half, p)
               : cudaLaunchKernelEx(&cfg, mla_partial_mh_kernel<false, false, true>, tm_pages, tm_kpe_half, p);
  if (bf16)
    return x16 ? cudaLaunchKernelEx(&cfg, mla_partial_mh_kernel<true, true, false>, tm_pages, tm_kpe_half, p)
               : cudaLaunchKernelEx(&cfg, mla_partial_mh_kernel<true, false, false>, tm_pages, tm_kpe_half, p);
  return x16 ? cudaLaunchKernelEx(&cfg, mla_partial_mh_kernel<false, true, false>, tm_pages, tm_kpe_half, p)
             : cudaLaunchKernelEx(&cfg, mla_partial_mh_kernel<false, false, false>, tm_pages, tm_kpe_half, p);
}

cudaError_t mh_read_clear_error(uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_device_error, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(uint32_t));
}

}  // namespace mla
