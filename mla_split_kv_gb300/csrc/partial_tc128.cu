// Tensor-core partial-decode kernel for CTAs of 16 query rows (fp16 or bf16)
// working in pairs, sm_103a.
//
// The operation is the one of the other partial kernels ("feat(core):
// matrix-absorbed MLA decode over a compressed-latent KV cache", *What
// changed*: SDPA(q_absorbed, ckv, ckv, scale, mask = scale * q_pe @ kpe^T),
// each chunk yielding a normalized partial and its log2 LSE).
//
// 16 query rows (the heads of a one-token decode) are too few for the tensor
// core's M side, so both products put tokens / latent columns on M=128 and the
// 16 rows on N:
//   S^T[tok, row] = [ckv | kpe][tok, :] . Q^T          M=128 tokens, N=16
//   O^T[d, row]  += ckv^T[d, tok] . P^T[tok, row]      M=128 columns, N=16, K=128
// At N=16 every tcgen05.mma costs about the same fixed time, so tiles are 128
// tokens (the most one M=128 instruction covers).
//
// A 128-token tile of the whole latent is 144 KB; it has to stay in shared
// memory from the score product until the PV product (after the softmax), and
// the next tiles have to be loading meanwhile, which does not fit in one SM.
// So the two CTAs of a pair (cluster ranks 2k, 2k+1) take the same tokens and
// split the latent columns: CTA `half` holds ckv columns [256 half, 256 half +
// 256) and kpe columns [32 half, 32 half + 32). Each computes a partial S^T
// over its columns, the two exchange them through distributed shared memory
// and add them (both get the same sum, in the same order), run the same
// softmax, and each accumulates O^T for its own 256 columns. A tile slot is
// then 72 KB (64 KB of ckv + 8 KB of kpe) and three fit, so tiles i+1 and i+2
// load while tile i is computed (a slot is held from its load through the
// score product, the exchange, the softmax and the PV product; with two slots
// the loads would wait on that whole chain). The kpe part of a slot is free
// once the tile's score product is done; it then takes the peer's partial
// scores of the tile, and after those are read, the tile's P^T. Pairs of a
// cluster split the chunk's tiles; the cluster combines at the end, in rank
// order. A chunk spread over several clusters skips that combine: every pair
// writes its part to the workspace and the last CTA to finish merges them.
//
// The ckv half of a tile arrives as one 4D TMA box per page (64 columns x 8
// rows x 4 column blocks x page/8 row groups): it lands as row groups of four
// swizzled [8 x 64] atoms, atom (g, c) at 4096 g + 1024 c. For the score MMAs
// (K-major, column block c) the 8-row groups are then 4 KB apart (SBO), and
// for the PV MMAs (MN-major, latent columns on M) the two 64-column blocks of
// an M=128 block are 1 KB apart (LBO) and the 8-token groups 4 KB (SBO). One
// TMA instruction per page and cache keeps the issue cost low.
//
// MMA order: as the inputs get ready, PV(j) first (it releases a slot), else
// S(i) (its tile landed and its TMEM buffer is free), each in tile order.
//
// Warp roles (384 threads, three warps per scheduler): warps 0-7 softmax / O
// rescale / epilogue (thread = token of the M=128 layout; the two warps of a
// TMEM lane quadrant take rows 0-7 and 8-15), warp 8 TMEM owner + MMA issuer,
// warps 9-11 producers (warp 9+k loads pages k, k+3, ... of each tile, both
// caches, one page per lane; the kpe box is this CTA's 32 columns, with the
// 64-byte swizzle). With three slots in flight an L2 prefetch of the next
// tile's pages measured slower over a sweep of caches larger than L2, so
// there is none. The kernel is a programmatic dependent launch: its set-up overlaps the
// end of the previous kernel in the stream.
#include "device_common.cuh"

namespace mla {

namespace {

constexpr int kT = 128;                          // tokens per tile
constexpr int kNR = 16;                          // query rows per CTA
constexpr int kHalfBoxes = 4;                    // ckv column blocks per CTA: 256 columns
constexpr int kHalfCols = kHalfBoxes * kBoxCols; // 256
constexpr int kKpeCols = kRope / 2;              // 32 rope columns per CTA
constexpr int kCkvBytes = kT * kHalfCols * 2;    // 64 KB: row group g, block c at 4096 g + 1024 c
constexpr int kKpeBytes = kT * kKpeCols * 2;     // 8 KB: [128 rows x 32 columns], 64-byte swizzle
constexpr int kTileSlot = kCkvBytes + kKpeBytes; // 72 KB
constexpr int kSlots = 3;
constexpr int kGroupBytes = 8 * kHalfCols * 2;   // 4 KB: one 8-row group of the four blocks
constexpr int kPageWarps = 3;                    // producer warps
constexpr int kSoftmaxWarps = 8;                 // two per TMEM lane quadrant: rows 0-7 and 8-15
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kMmaWarp = kSoftmaxWarps;
constexpr int kThreads = (kSoftmaxWarps + 1 + kPageWarps) * 32;  // 384: three warps per scheduler
constexpr int kRH = kNR / 2;                     // rows per softmax thread
constexpr int kMaxPagesPerWarp = (kT / 16 + kPageWarps - 1) / kPageWarps;  // pages of 16 tokens or more
constexpr float kRescaleTau = 8.0f;
// E4M3 caches: a tile's bytes land unswizzled in the upper half of its slot (staged rows of 256
// bytes: ckv tokens 0-127, then the kpe, 8 tokens a row) and are widened to fp16 in place.
constexpr int kStage = kTileSlot - kT * (kHalfCols + kKpeCols);  // 36 KB
constexpr int kStageRows = kT * (kHalfCols + kKpeCols) / kHalfCols;  // 144
static_assert(kStage == 9 * kGroupBytes && kStageRows == 144 && kCkvBytes == kStage + 112 * kHalfCols,
              "the widening order below assumes this geometry");

constexpr uint32_t kOffTile = 0;                            // 3 tile slots
constexpr uint32_t kOffQ = kSlots * kTileSlot;              // 216 KB: Q^T
constexpr uint32_t kQChunk = kNR * 128;                     // [16 x 64] fp16, 128-byte swizzle: 2 KB
constexpr uint32_t kQKpe = kNR * kKpeCols * 2;              // [16 x 32] fp16, 64-byte swizzle: 1 KB
constexpr uint32_t kOffSmall = kOffQ + kHalfBoxes * kQChunk + kQKpe;  // 225 KB
constexpr uint32_t kSmallBytes = 1024;
// no alignment slack: the dynamic shared memory of a CTA starts 1024-byte aligned (checked at run
// time), and at 226 KB a CTA of the entries merge kernel (no shared memory) still fits on the SM
constexpr uint32_t kSmem = kOffSmall + kSmallBytes;
// in the kpe part of a slot, after the tile's score product: the peer's partial S, then P^T
constexpr uint32_t kXBuf = kNR * kT * 4;                    // [128 tokens][16 rows] fp32: 8 KB
constexpr uint32_t kPBytes = 2 * kNR * 128;                 // P^T [16 x 128 tokens]: two 64-token atoms
// (bf16: P^T as two bf16 terms, hi then lo, 2 x kPBytes: the whole kpe part of the slot)
constexpr uint32_t kTmemCols = 64;                          // S^T 2 x 16 + O^T 2 x 16
static_assert(kSmem <= 232448, "shared memory per CTA");
static_assert(kXBuf <= kKpeBytes && 2 * kPBytes <= kKpeBytes, "exchange and P^T (hi, lo) fit the kpe part of a slot");
static_assert(kCkvBytes % 1024 == 0 && kTileSlot % 1024 == 0, "swizzle atoms stay aligned");
static_assert(kNR * kHalfCols * 4 + 2 * kNR * 4 <= kSlots * kTileSlot, "epilogue staging fits the tile slots");

struct Small {
  // slot ring: full / empty; TMEM S buffers (tile parity): sfull / sfree; per slot: ppfull (P^T
  // written), xfull (the peer's partial S landed), xready (the peer's score product of the slot's
  // tile is done: its kpe part is free for this CTA's partial S); pvdone per tile parity
  uint64_t full[kSlots], empty[kSlots], sfull[2], sfree[2], ppfull[kSlots], pvdone[2], xfull[kSlots],
      xready[kSlots], drain;
  // E4M3 caches: the bytes of a tile landed in its slot (TMA), and the producer warps' meeting point
  // inside each tile's in-place conversion (one phase per tile)
  uint64_t landed[kSlots], conv;
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t last_cluster;  // this CTA took the last ticket of its chunk half (spread plans)
  int32_t last_request;  // this CTA took the last ticket of its request slice (single-launch decode)
  float red[4][kNR];
  float mref[kNR];
  float alpha[kNR];
};
static_assert(sizeof(Small) <= kSmallBytes, "small smem region");

__device__ __forceinline__ uint32_t tmem_lane_base(int warp) { return static_cast<uint32_t>(32 * (warp & 3)) << 16; }

// kFp8: E4M3 caches (byte loads, widened in the slot, cache scale on the output); kBf16: bf16 queries and
// caches (the probabilities carried as two bf16 terms, two PV products a step); one instance each
template <bool kFp8, bool kBf16>
__global__ void __launch_bounds__(kThreads, 1)
    mla_partial_tc128_kernel(const __grid_constant__ CUtensorMap tm_pages, const __grid_constant__ CUtensorMap tm_kpe_half,
                             const PartialParams p) {
  extern __shared__ uint8_t smem_raw[];
  // the swizzled tile and Q layouts need a 1024-byte aligned base, and the size leaves no slack to
  // align it: a launch that breaks this (it does not happen on sm_103a) flags it and does nothing
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) flag_error(MLA_DEVERR_CONFIG);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* qs = smem + kOffQ;
  Small* sm = reinterpret_cast<Small*>(smem + kOffSmall);
  volatile int32_t* abort_flag = &sm->abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank(), nranks = cluster_nctarank(), peer = rank ^ 1u;
  const int half = static_cast<int>(rank & 1u);
  // a chunk may be spread over `subs` clusters (grid.y = chunk * subs + sub); its tiles are
  // split over all their pairs
  const int subs = (p.subs > 1) ? p.subs : 1;
  const int chunk = static_cast<int>(blockIdx.y) / subs, sub = static_cast<int>(blockIdx.y) % subs;
  const int cluster_pairs = static_cast<int>(nranks >> 1);
  const int rows_total = p.q_len * p.H;

  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&sm->full[s], kPageWarps);  // one expect_tx arrival per producer warp
      mbar_init(&sm->empty[s], 1);
      mbar_init(&sm->ppfull[s], kSoftmaxWarps);
      mbar_init(&sm->xfull[s], 1);   // local expect_tx arrival + the peer's st.async bytes
      mbar_init(&sm->xready[s], 1);  // the peer's MMA commit
      mbar_init(&sm->landed[s], kPageWarps);
    }
    mbar_init(&sm->conv, kPageWarps);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm->sfull[t], 1);
      mbar_init(&sm->sfree[t], kSoftmaxWarps);
      mbar_init(&sm->pvdone[t], 1);
    }
    mbar_init(&sm->drain, 1);
    sm->abort_flag = 0;
    fence_mbar_init();
  }
  if (tid < kNR) sm->mref[tid] = -INFINITY;
  if (warp == kMmaWarp) {
    tmem_alloc(&sm->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive_release();  // the peer touches this CTA's barriers only after this cluster phase
  const uint32_t tmem = sm->tmem_base;
  // Launched as a programmatic dependent of the previous kernel in the stream: the set-up above
  // overlaps its end. The queries and the caches are read after the wait below; so are the chunk
  // table, the lengths and the block table, unless the caller declared them complete before that
  // kernel started (tables_ready): then they are read while it finishes (producers: the first
  // block-table window too). The next kernel (the merge) is released only after the wait, so a
  // kernel launched after this one starts once everything before this one has finished.
  CtaWork w{};
  const int pair_index = sub * cluster_pairs + static_cast<int>(rank >> 1);
  int win_base = -1, win_pid = -1;  // producers: a window of 32 block-table entries (page ids)
  auto load_window = [&](int pg) {   // warp-uniform page index
    win_base = pg & ~31;
    const int q = win_base + lane;
    const int npages_req = (w.L + p.bs - 1) / p.bs;
    win_pid = (q < npages_req && q < p.max_blocks) ? checked_page(p, w.b, q) : -1;
  };
  // producers: warp kMmaWarp + 1 + k0 loads pages k0, k0 + kPageWarps, ... of each tile
  const int k0 = warp - kMmaWarp - 1;
  auto page_of = [&](int pg) -> int {  // warp-uniform pg
    if ((pg & ~31) != win_base) load_window(pg);
    return __shfl_sync(0xffffffffu, win_pid, pg & 31);
  };
  // the physical pages of this warp's share of tile i (block-table reads); returns their number
  auto tile_pids = [&](int i, int* pids) -> int {
    const int tok0 = w.sub0 + i * kT;
    const int pg0 = tok0 / p.bs;
    const int npg = (min(kT, w.sub1 - tok0) + p.bs - 1) / p.bs;
    const int mine = (npg > k0) ? (npg - k0 + kPageWarps - 1) / kPageWarps : 0;
#pragma unroll
    for (int m = 0; m < kMaxPagesPerWarp; ++m) pids[m] = (m < mine) ? page_of(pg0 + k0 + m * kPageWarps) : -1;
    return mine;
  };
  // the loads of those pages into the slot of tile i (free), counted on its full barrier; lane m
  // issues page m (TMA issue from several lanes overlaps)
  auto tile_issue = [&](int i, const int* pids, int mine, uint64_t pol) {
    const int s = i % kSlots;
    uint8_t* slot = smem + kOffTile + s * kTileSlot;
    if (kFp8) {
      // E4M3 bytes, unswizzled, into the upper half of the slot: ckv rows of 256 bytes, then kpe rows of 32
      if (lane == 0) mbar_arrive_expect_tx(&sm->landed[s], static_cast<uint32_t>(mine * p.bs * (kHalfCols + kKpeCols)));
      __syncwarp();
#pragma unroll
      for (int m = 0; m < kMaxPagesPerWarp; ++m) {
        if (lane == m && m < mine) {
          const int j = k0 + m * kPageWarps;  // page of the tile
          tma_load_2d(slot + kStage + j * p.bs * kHalfCols, &tm_pages, kHalfCols * half, pids[m] * p.bs,
                      &sm->landed[s], pol);
          tma_load_2d(slot + kStage + kT * kHalfCols + j * p.bs * kKpeCols, &tm_kpe_half, kKpeCols * half,
                      pids[m] * p.bs, &sm->landed[s], pol);
        }
      }
      return;
    }
    if (lane == 0) mbar_arrive_expect_tx(&sm->full[s], static_cast<uint32_t>(mine * p.bs * (kHalfCols + kKpeCols) * 2));
    __syncwarp();
#pragma unroll
    for (int m = 0; m < kMaxPagesPerWarp; ++m) {
      if (lane == m && m < mine) {
        const int j = k0 + m * kPageWarps;  // page of the tile
        tma_load_4d(slot + j * p.bs * (kHalfCols * 2), &tm_pages, 0, 0, kHalfBoxes * half, pids[m] * (p.bs / 8),
                    &sm->full[s], pol);
        tma_load_2d(slot + kCkvBytes + j * p.bs * (kKpeCols * 2), &tm_kpe_half, kKpeCols * half, pids[m] * p.bs,
                    &sm->full[s], pol);
      }
    }
  };
  // E4M3 caches: tile i's staged bytes become the 16-bit tile in place, in the layouts the 16-bit loads
  // give (ckv: 128-byte-swizzled [8 x 64] atoms, a 4 KB row group per 8 tokens; kpe: 64-byte
  // swizzle), by the three producer warps. A warp step takes two staged rows (512 bytes, 16 a lane):
  // ckv tokens t, t+1 (t even), or 16 kpe tokens. The 16-bit rows of ckv tokens 0-71 lie below the
  // staging; those of tokens 8g..8g+7 (g >= 9) overwrite staged rows 16(g-9)..16(g-9)+15, and the
  // 16-bit kpe staged rows 112-143. So, with the three warps meeting between the parts: tokens 0-71 |
  // tokens 72-103, then staged rows 104-143 into registers | those rows (tokens 104-127, the kpe) from
  // the registers. Every staged row is read before a part that overwrites it. Lane 0 of each warp
  // then counts it on the slot's full barrier.
  // ckv lanes: quarter q and half r2 of it take token t + r2, column block q ^ r2, 16 columns 16 (lane
  // & 3) .. +15 (8-column pieces 2 (lane & 3), +1): the 8 lanes of a quarter read 8 different 16-byte
  // bank groups and, the two halves writing rows of opposite parity, write 8 different ones
  const int r2 = (lane >> 2) & 1, cbl = (lane >> 3) ^ r2, kk = lane & 3;
  const int src_ckv = r2 * kHalfCols + cbl * 64 + kk * 16;  // in the two staged rows of a step
  // kpe lanes: token 16 j + lane / 2 of step j, fp8 columns 16 (lane & 1) .. +15
  const int tk_l = lane >> 1, hk = lane & 1;
  auto ckv_store = [&](uint32_t slot, int t, const uint4 v) {  // ckv tokens t + r2 (t even)
    const int r = (t & 7) + r2;
    const uint32_t row = slot + (t >> 3) * kGroupBytes + cbl * 1024 + r * 128;
    widen16(v, row + (((2 * kk) ^ r) << 4), row + (((2 * kk + 1) ^ r) << 4));
  };
  auto kpe_store = [&](uint32_t slot, int j, const uint4 v) {  // kpe step j: tokens 16 j .. 16 j + 15
    const int tk = 16 * j + tk_l;
    const uint32_t row = slot + kCkvBytes + tk * (kKpeCols * 2);
    widen16(v, row + ((((2 * hk) ^ (tk >> 1)) & 3) << 4), row + ((((2 * hk + 1) ^ (tk >> 1)) & 3) << 4));
  };
  // the three producer warps meet (two phases per tile); the wait spins rather than suspends, the
  // others being at most a few hundred cycles away
  auto meet = [&](int phase) -> bool {
    __syncwarp();
    int ok = 1;
    if (lane == 0) {
      mbar_arrive(&sm->conv);
      if (!mbar_test(&sm->conv, phase & 1)) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_test(&sm->conv, phase & 1)) {
          if (globaltimer_ns() - t0 > p.timeout_ns) {
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
    if (!__all_sync(0xffffffffu, mbar_wait(&sm->landed[s], (i / kSlots) & 1, p.timeout_ns))) return false;
    widen_ckv_steps(slot, stage_src, 2 * k0, 12, r2, cbl, kk);  // tokens 0-71: 36 steps, 12 a warp
    if (!meet(2 * i)) return false;
    widen_ckv_steps(slot, stage_src, 72 + 2 * k0, k0 == 0 ? 6 : 5, r2, cbl, kk);  // 72-103: 6, 5, 5
    // staged rows 104-143 in 20 steps (7, 7, 6): steps 0-11 ckv tokens 104-127, steps 12-19 the kpe
    constexpr int kHeld = 7;
    uint4 held[kHeld];
#pragma unroll
    for (int m = 0; m < kHeld; ++m) {
      const int j = k0 + kPageWarps * m;
      if (j < 20) held[m] = lds128(slot + kStage + (104 + 2 * j) * kHalfCols + (j < 12 ? src_ckv : lane * 16));
    }
    if (!meet(2 * i + 1)) return false;
#pragma unroll
    for (int m = 0; m < kHeld; ++m) {
      const int j = k0 + kPageWarps * m;
      if (j < 12)
        ckv_store(slot, 104 + 2 * j, held[m]);
      else if (j < 20)
        kpe_store(slot, j - 12, held[m]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm->full[s]);
    return true;
  };
  int issued = -1;  // producers: the last tile whose loads this warp issued
  if (p.tables_ready) {
    w = cta_work(p, kNR, kT, pair_index, subs * cluster_pairs, chunk);
    if (warp > kMmaWarp && w.sub1 > w.sub0) load_window(w.sub0 / p.bs);
  }
  // the tensor-map descriptors are kernel parameters, not data of the preceding kernel: fetch them
  // now, so the first page loads do not pay for it
  if (warp == kMmaWarp + 1 && lane == 0) {
    tma_prefetch_desc(&tm_pages);
    tma_prefetch_desc(&tm_kpe_half);
  }
  // prefix_ready: the cache rows before each request's window are final before the preceding kernel
  // ends, so the first tiles (one per slot) whose tokens all lie before the window are loaded while
  // it finishes; the window's own rows (which that kernel may be writing) only after the wait
  if (p.prefix_ready && p.tables_ready && warp > kMmaWarp) {
    const uint64_t pol = l2_policy_evict_first();
    const int n = (w.sub1 - w.sub0 + kT - 1) / kT;
    const int before = w.L - p.q_len;  // first position of the window
    for (int i = 0; i < min(n, kSlots); ++i) {
      if (min(w.sub0 + (i + 1) * kT, w.sub1) > before) break;
      int pids[kMaxPagesPerWarp];
      const int mine = tile_pids(i, pids);
      tile_issue(i, pids, mine, pol);
      issued = i;
    }
  }
  pdl_wait();
  pdl_launch_dependents();  // the merge of these partials may be scheduled now; it waits for this grid
  if (!p.tables_ready) w = cta_work(p, kNR, kT, pair_index, subs * cluster_pairs, chunk);
  const int ntiles = (w.sub1 - w.sub0 + kT - 1) / kT;
  // single-launch decode: request b's chunk slots, whose partials this launch also merges
  const bool fused = p.out != nullptr;  // the TICKETS way of mla_decode
  int req_lo = 0, req_hi = 0;
  if (fused && w.b >= 0 && w.b < p.B) request_slots(p, w.b, &req_lo, &req_hi);

  if (warp > kMmaWarp) {
    // ------------------------------------------------------------------ producers
    const uint64_t pol = l2_policy_evict_first();
    if (kFp8) {
      // Issue and widening interleave: the next tile's loads as soon as its slot is free, else the
      // widening of the oldest landed tile; nothing to do for longer than the wait limit (or an abort
      // elsewhere) ends it
      int ni = issued + 1, nc = 0;
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
            } else if (now - idle_t0 > p.timeout_ns) {
              act = -1;
              *abort_flag = 1;
              flag_error(MLA_DEVERR_TIMEOUT);
            }
          }
          if (act > 0) idle = false;
        }
        act = __shfl_sync(0xffffffffu, act, 0);
        if (act == 1) {
          int pids[kMaxPagesPerWarp];
          const int mine = tile_pids(ni, pids);
          tile_issue(ni, pids, mine, pol);
          issued = ni++;
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
    }
    for (int i = kFp8 ? ntiles : issued + 1; i < ntiles; ++i) {
      const int s = i % kSlots;
      // the pages of tile i first: their block-table reads overlap the wait for the slot
      int pids[kMaxPagesPerWarp];
      const int mine = tile_pids(i, pids);
      if (i >= kSlots) {  // tile i-3 released the slot
        int ok = 1;
        if (lane == 0) {
          ok = mbar_wait(&sm->empty[s], ((i / kSlots) - 1) & 1, p.timeout_ns) && !*abort_flag;
          if (!ok) *abort_flag = 1;
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
      tile_issue(i, pids, mine, pol);
      issued = i;
    }
    // after an abort, let this warp's loads still in flight (the last three tiles it issued, one per
    // slot) land before shared memory is released
    if (lane == 0 && *abort_flag)
      for (int t = max(0, issued - (kSlots - 1)); t <= issued; ++t)
        mbar_wait(kFp8 ? &sm->landed[t % kSlots] : &sm->full[t % kSlots], (t / kSlots) & 1, kDrainTimeoutNs);
    cluster_wait_acquire();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    const uint32_t idesc_s = idesc_f16_f32(128, kNR, kBf16, false, false);
    const uint32_t idesc_o = idesc_f16_f32(128, kNR, kBf16, true, false);
    const Desc2 qd = desc2(smem_desc_sw128(smem_u32(qs), 16, 1024));
    const Desc2 qk = desc2(smem_desc_sw64(smem_u32(qs + kHalfBoxes * kQChunk), 512));
    const uint32_t tile_base = smem_u32(smem + kOffTile);
    uint64_t tmo = p.timeout_ns;
    asm volatile("" : "+l"(tmo));
    // score product of tile i (slot i % 3) into S buffer i & 1: this CTA's 4 ckv column blocks,
    // then its 32 kpe columns (two K steps of the 64-byte-swizzled box)
    auto score = [&](int i) {
      const int t = i & 1;
      if (lane == 0) {
        tc_fence_after();
        const uint32_t slot = tile_base + (i % kSlots) * kTileSlot;
        const Desc2 ad = desc2(smem_desc_sw128(slot, 16, kGroupBytes));
        const Desc2 ak = desc2(smem_desc_sw64(slot + kCkvBytes, 512));
        const uint32_t d = tmem + t * kNR;
#pragma unroll
        for (int c = 0; c < kHalfBoxes; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ss(d, ad, (c * 1024 + kk * 32) >> 4, qd, (c * kQChunk + kk * 32) >> 4, idesc_s,
                    (c == 0 && kk == 0) ? 0u : 1u);
        umma_ss(d, ak, 0, qk, 0, idesc_s, 1u);
        umma_ss(d, ak, 32 >> 4, qk, 32 >> 4, idesc_s, 1u);
        umma_commit(&sm->sfull[t]);
        // once these MMAs have read the kpe part of the slot, the peer may send its partial scores there
        umma_commit_multicast(&sm->xready[i % kSlots], static_cast<uint16_t>(1u << peer));
      }
      __syncwarp();
    };
    // rows [nvalid, nend) of the ckv part of a slot: zero them so the PV operand stays finite
    // (the probabilities there are 0, but stale or unwritten rows may hold non-finite values)
    auto zero_rows = [&](uint8_t* ckv, int nvalid, int nend) {
      for (int x = lane; x < (nend - nvalid) * kHalfBoxes * 8; x += 32) {
        const int rc = x >> 3, tok = nvalid + rc / kHalfBoxes, c = rc % kHalfBoxes;
        *reinterpret_cast<uint4*>(ckv + (tok >> 3) * kGroupBytes + c * 1024 + (tok & 7) * 128 + (x & 7) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
    };
    // PV product of tile i: O^T rows [128 blk, 128 blk + 128) of this CTA's columns = boxes 2 blk,
    // 2 blk + 1; P^T is in the kpe part of the tile's slot
    auto pv = [&](int i) {
      const int s = i % kSlots, t = i & 1;
      const int nvalid = min(kT, w.sub1 - (w.sub0 + i * kT));
      // K steps of 16 tokens that hold valid tokens; in a partial tile only the rows up to the
      // next multiple of 16 are read, and those past the end are zeroed (the score product of
      // tile i is complete: its softmax ran)
      const int ksteps = (nvalid + 15) >> 4;
      if (nvalid < (ksteps << 4)) {
        zero_rows(smem + kOffTile + s * kTileSlot, nvalid, ksteps << 4);
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        tc_fence_after();
        const uint32_t slot = tile_base + s * kTileSlot;
        const Desc2 pb = desc2(smem_desc_sw128(slot + kCkvBytes, 16, 1024));
        const uint32_t acc0 = (i > 0) ? 1u : 0u;
        // K step ks: tokens [16 ks, 16 ks + 16): two 8-token groups of the slot, and 16 tokens of the
        // P^T atom (ks / 4) at 32-byte step ks % 4
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          const Desc2 a0 = desc2(smem_desc_sw128(slot + 2 * blk * 1024, 1024, kGroupBytes));
          const uint32_t d = tmem + 2 * kNR + blk * kNR;
          if (ksteps == kT / 16) {
#pragma unroll
            for (int ks = 0; ks < kT / 16; ++ks) {
              umma_ss(d, a0, (ks * 2 * kGroupBytes) >> 4, pb, ((ks >> 2) * (kNR * 128) + (ks & 3) * 32) >> 4, idesc_o,
                      ks > 0 ? 1u : acc0);
              if (kBf16)  // the lo term of the probabilities, kPBytes further
                umma_ss(d, a0, (ks * 2 * kGroupBytes) >> 4, pb,
                        (kPBytes + (ks >> 2) * (kNR * 128) + (ks & 3) * 32) >> 4, idesc_o, 1u);
            }
          } else {
            for (int ks = 0; ks < ksteps; ++ks) {
              umma_ss(d, a0, (ks * 2 * kGroupBytes) >> 4, pb, ((ks >> 2) * (kNR * 128) + (ks & 3) * 32) >> 4, idesc_o,
                      ks > 0 ? 1u : acc0);
              if (kBf16)
                umma_ss(d, a0, (ks * 2 * kGroupBytes) >> 4, pb,
                        (kPBytes + (ks >> 2) * (kNR * 128) + (ks & 3) * 32) >> 4, idesc_o, 1u);
            }
          }
        }
        umma_commit(&sm->empty[s]);
        umma_commit(&sm->pvdone[t]);
      }
      __syncwarp();
    };
    named_bar_sync(2, kSoftmaxThreads + 32);  // Q^T staged by the softmax warps
    cluster_wait_acquire();                   // the peer's barriers are initialised (commits reach them)
    // Issue as the inputs get ready, each product in tile order: PV(np) once P^T(np) is written
    // (first: it releases a slot for the next load), else S(ns) once tile ns has landed and its S
    // buffer is free. Nothing ready for longer than the wait limit (or an abort elsewhere) ends it.
    int ns = 0, np = 0;
    bool idle = false;
    uint64_t idle_t0 = 0;
    while (np < ntiles) {
      int act = 0;
      if (lane == 0) {
        if (np < ns && mbar_test(&sm->ppfull[np % kSlots], (np / kSlots) & 1)) {
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
  } else {
    // ------------------------------------------------------------------ softmax (warps 0-7)
    // kernel parameters used every tile, held in registers (not re-read from the parameter bank)
    float scale_log2 = p.scale_log2;
    uint64_t tmo = p.timeout_ns;
    asm volatile("" : "+f"(scale_log2), "+l"(tmo));
    // Q^T: this CTA's 256 latent columns (4 chunks, 128-byte swizzle), then its 32 kpe columns
    // (one chunk, 64-byte swizzle); 16 rows, K-major
    // (every thread's loads are issued before its shared-memory stores: one round trip, not three)
    constexpr int kQPieces = (kHalfCols + kKpeCols) / 8;  // 16-byte pieces per row
    constexpr int kQIters = (kNR * kQPieces + kSoftmaxThreads - 1) / kSoftmaxThreads;
    uint4 qv[kQIters];
#pragma unroll
    for (int it = 0; it < kQIters; ++it) {
      const int idx = tid + it * kSoftmaxThreads;
      const int r = idx / kQPieces, k = (idx % kQPieces) * 8;
      qv[it] = make_uint4(0u, 0u, 0u, 0u);
      if (idx < kNR * kQPieces && r < w.nrows) {
        const long long row = static_cast<long long>(w.b) * rows_total + w.row0 + r;
        qv[it] = (k < kHalfCols)
                     ? __ldcg(reinterpret_cast<const uint4*>(p.q_abs + row * kRank + kHalfCols * half + k))
                     : __ldcg(reinterpret_cast<const uint4*>(p.q_pe + row * kRope + kKpeCols * half + (k - kHalfCols)));
      }
    }
#pragma unroll
    for (int it = 0; it < kQIters; ++it) {
      const int idx = tid + it * kSoftmaxThreads;
      if (idx >= kNR * kQPieces) break;
      const int r = idx / kQPieces, k = (idx % kQPieces) * 8;
      uint8_t* dst = (k < kHalfCols) ? qs + (k / kBoxCols) * kQChunk + sw128_offset(r, k % kBoxCols)
                                     : qs + kHalfBoxes * kQChunk + sw64_offset(r, k - kHalfCols);
      *reinterpret_cast<uint4*>(dst) = qv[it];
    }
    fence_proxy_async_smem();
    named_bar_arrive(2, kSoftmaxThreads + 32);
    cluster_wait_acquire();  // the peer's barriers are initialised

    // Thread (warp, lane) owns token tl = 32 (warp % 4) + lane of each tile (M=128 layout of S^T)
    // and rows [8 h, 8 h + 8), h = warp / 4 (the two warps of a TMEM lane quadrant split the rows).
    const int q4 = warp & 3, h = warp >> 2;
    const int tl = 32 * q4 + lane;
    const uint32_t lane_base = tmem_lane_base(q4);
    float lsum[kRH], mr[kRH];  // running row sums over this thread's tokens; reference max per row
#pragma unroll
    for (int k = 0; k < kRH; ++k) {
      lsum[k] = 0.f;
      mr[k] = -INFINITY;
    }
    const int causal_floor = p.causal ? w.L - p.q_len + w.row0 / p.H : 0x7fffffff;
    // the peer's partial S of a tile, in the kpe part of the tile's slot, [token][16 rows] fp32: row
    // tl's 16 values are 4 float4 chunks, chunk c at position c ^ ((tl >> 1) & 3) (conflict-free
    // 16-byte accesses); this thread's rows are chunks 2h, 2h+1
    const uint32_t xsw = static_cast<uint32_t>((tl >> 1) & 3);
    const uint32_t peer_x = dsmem_addr(smem + kOffTile + kCkvBytes, peer) + tl * 64;  // + slot * kTileSlot
    bool ok_all = true;
    // A(i), first part, which never waits on the peer: the expectation of the peer's partial scores
    // of tile i in the kpe part of the slot (the completion of this CTA's score product tells the
    // peer that it may send them; the bytes may land before this), then this warp's partial scores
    // of tile i (and its S buffer freed).
    auto prep = [&](int i, float* x) -> bool {
      const int b = i & 1, s = i % kSlots;
      if (warp == 0 && lane == 0) mbar_arrive_expect_tx(&sm->xfull[s], kXBuf);
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&sm->sfull[b], (i >> 1) & 1, tmo);
      if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
      tc_fence_after();
      tmem_ld8(tmem + lane_base + b * kNR + kRH * h, x);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->sfree[b]);
      return true;
    };
    // the peer's score product of tile i is done, so tile i's scores may go to its slot
    // (non-blocking test)
    auto peer_free = [&](int i) -> bool {
      int ready = 0;
      if (lane == 0) ready = mbar_test(&sm->xready[i % kSlots], (i / kSlots) & 1) ? 1 : 0;
      return __shfl_sync(0xffffffffu, ready, 0) != 0;
    };
    // A(i), second part: once the peer's score product of tile i is done, this warp's partial scores
    // of tile i go to the kpe part of the peer's slot
    auto push = [&](int i, const float* x) -> bool {
      const int s = i % kSlots;
      const int ok = mbar_wait_cluster(&sm->xready[s], (i / kSlots) & 1, tmo);
      if (!__all_sync(0xffffffffu, ok)) return false;
      const uint32_t dst = peer_x + s * kTileSlot;
      const uint32_t rbar = dsmem_addr(&sm->xfull[s], peer);
#pragma unroll
      for (int c = 0; c < 2; ++c)
        dsmem_st_async_f32x4(dst + (((2 * h + c) ^ xsw) << 4),
                             make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]), rbar);
      return true;
    };
    // B(i): add the peer's part, scale and mask, lazy rescale, probabilities -> P^T. Every softmax
    // warp calls it for every tile it reaches, also after a failed send (sent = false), so all of
    // them pass the same named barriers; a failure anywhere ends the loop in all of them.
    auto finish = [&](int i, float* x, bool sent) -> bool {
      const int s = i % kSlots;
      uint8_t* region = smem + kOffTile + s * kTileSlot + kCkvBytes;  // the peer's partial S, then P^T
      const int tok0 = w.sub0 + i * kT;
      const int nvalid = min(kT, w.sub1 - tok0);
      const bool masked_tile = (nvalid < kT) || (tok0 + kT - 1 > causal_floor) || (w.nrows < kNR);
      int ok = sent ? mbar_wait_cluster(&sm->xfull[s], (i / kSlots) & 1, tmo) : 0;
      ok = __all_sync(0xffffffffu, ok);
      bool need_local = false;
      if (ok) {
        const float4* xb = reinterpret_cast<const float4*>(region) + tl * 4;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const float4 y = xb[(2 * h + c) ^ xsw];
          // rank-0 part + rank-1 part, the same sum in both CTAs
          x[4 * c] = half ? (y.x + x[4 * c]) : (x[4 * c] + y.x);
          x[4 * c + 1] = half ? (y.y + x[4 * c + 1]) : (x[4 * c + 1] + y.y);
          x[4 * c + 2] = half ? (y.z + x[4 * c + 2]) : (x[4 * c + 2] + y.z);
          x[4 * c + 3] = half ? (y.w + x[4 * c + 3]) : (x[4 * c + 3] + y.w);
        }
        if (__builtin_expect(masked_tile, 0)) {  // tail of the chunk, causal edge, or fewer than 16 rows
          const int t = tok0 + tl;
#pragma unroll
          for (int k = 0; k < kRH; ++k) {
            const int r = kRH * h + k;
            bool vis = (tl < nvalid) && (r < w.nrows);
            if (p.causal) vis = vis && (t <= w.L - p.q_len + (w.row0 + r) / p.H);
            x[k] = vis ? x[k] * scale_log2 : -INFINITY;
          }
        } else {
#pragma unroll
          for (int k = 0; k < kRH; ++k) x[k] *= scale_log2;
        }
#pragma unroll
        for (int k = 0; k < kRH; ++k) need_local |= x[k] > mr[k] + kRescaleTau;
      } else {
#pragma unroll
        for (int k = 0; k < kRH; ++k) x[k] = -INFINITY;
        *abort_flag = 1;
      }
      if (__builtin_expect(named_bar_sync_or(1, kSoftmaxThreads, need_local || !ok || *abort_flag != 0), 0)) {
        if (named_bar_sync_or(1, kSoftmaxThreads, *abort_flag != 0)) return false;
        // rare path: move the reference max, rescale O^T and the row sums
#pragma unroll
        for (int k = 0; k < kRH; ++k) {
          float v = x[k];
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
          if (lane == 0) sm->red[q4][kRH * h + k] = v;
        }
        named_bar_sync(1, kSoftmaxThreads);
        if (tid < kNR) {
          const float mprev = sm->mref[tid];
          const float tmax = fmaxf(fmaxf(sm->red[0][tid], sm->red[1][tid]), fmaxf(sm->red[2][tid], sm->red[3][tid]));
          const float mnew = fmaxf(mprev, tmax);
          sm->alpha[tid] = (mnew == -INFINITY) ? 1.f : exp2f(mprev - mnew);
          sm->mref[tid] = mnew;
        }
        named_bar_sync(1, kSoftmaxThreads);
#pragma unroll
        for (int k = 0; k < kRH; ++k) mr[k] = sm->mref[kRH * h + k];
        if (i >= 1) {  // PV(i-1) must be complete before O^T is rescaled
          int ok2 = 1;
          if (lane == 0) ok2 = mbar_wait(&sm->pvdone[(i - 1) & 1], ((i - 1) >> 1) & 1, tmo);
          if (__shfl_sync(0xffffffffu, ok2, 0)) {
            tc_fence_after();
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
              float v[kRH];
              const uint32_t a = tmem + lane_base + 2 * kNR + blk * kNR + kRH * h;
              tmem_ld8(a, v);
              tmem_wait_ld();
#pragma unroll
              for (int k = 0; k < kRH; ++k) v[k] *= sm->alpha[kRH * h + k];
              tmem_st8(a, v);
            }
            tmem_wait_st();
          } else if (lane == 0) {
            *abort_flag = 1;
          }
        }
#pragma unroll
        for (int k = 0; k < kRH; ++k) lsum[k] *= sm->alpha[kRH * h + k];
      }
      {  // probabilities -> P^T (16-bit, K-major, two swizzled 64-token atoms; bf16: a second P^T of the
         // rounding remainders kPBytes further) and row sums, over the peer's partial S (every softmax
         // warp has read its part: the barrier above)
        uint8_t* pb = region + (tl >> 6) * (kNR * 128);
#pragma unroll
        for (int k = 0; k < kRH; ++k) {
          // masked scores (-inf) give 0; a row with no visible token yet subtracts a finite stand-in
          const float pr = fast_exp2(x[k] - ((mr[k] == -INFINITY) ? 0.f : mr[k]));
          const uint16_t hv = f2h<kBf16>(pr);
          const uint32_t off = sw128_offset(kRH * h + k, tl & 63);
          *reinterpret_cast<uint16_t*>(pb + off) = hv;
          if (kBf16) {
            const float hf = h2f<true>(hv);
            const uint16_t lv = f2h<true>(pr - hf);
            lsum[k] += hf + h2f<true>(lv);
            *reinterpret_cast<uint16_t*>(pb + kPBytes + off) = lv;
          } else {
            lsum[k] += h2f<false>(hv);
          }
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->ppfull[s]);
      return true;
    };
    // Tile by tile, one ahead: when tile i+1's scores are already there, they are loaded (and, if the
    // peer's buffer is already free, sent) before tile i is finished, so the exchange of one overlaps
    // the work on the other; otherwise tile i is finished first, so PV(i) is not held back. Each warp
    // decides for itself, so no warp may wait on the peer between the two: the peer's warps that
    // would release it may be held at their own barrier in B(i) by their warps that are waiting on
    // this CTA the same way.
    {
      float xc[kRH], xn[kRH];  // tile i's scores; tile i+1's, when loaded early
      bool c_prepped = false, c_sent = false;
      for (int i = 0; i < ntiles && ok_all; ++i) {
        if (!c_prepped) c_prepped = prep(i, xc);
        if (c_prepped && !c_sent) c_sent = push(i, xc);
        bool n_prepped = false, n_sent = false;
        if (c_sent && i + 1 < ntiles) {
          int ready = 0;
          if (lane == 0) ready = mbar_test(&sm->sfull[(i + 1) & 1], ((i + 1) >> 1) & 1) ? 1 : 0;
          if (__shfl_sync(0xffffffffu, ready, 0) != 0) {
            n_prepped = prep(i + 1, xn);
            if (n_prepped && peer_free(i + 1)) n_sent = push(i + 1, xn);
          }
        }
        ok_all = finish(i, xc, c_sent);
#pragma unroll
        for (int k = 0; k < kRH; ++k) xc[k] = xn[k];
        c_prepped = n_prepped;
        c_sent = n_sent;
      }
    }
    if (!ok_all && lane == 0) *abort_flag = 1;
    const bool aborted = named_bar_sync_or(1, kSoftmaxThreads, *abort_flag != 0);
    if (ntiles > 0 && !aborted) {
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&sm->pvdone[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, tmo);
      if (!__shfl_sync(0xffffffffu, ok, 0) && lane == 0) *abort_flag = 1;
    }
#pragma unroll
    for (int k = 0; k < kRH; ++k) {
      float v = lsum[k];
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      if (lane == 0) sm->red[q4][kRH * h + k] = v;
    }
    named_bar_sync(1, kSoftmaxThreads);
  }
  __syncthreads();  // all roles done: the tile slots are free for staging
  const bool have = (ntiles > 0) && !*abort_flag;
  if (subs > 1 || p.entries_only) {
    // A chunk spread over several clusters (or any chunk when the merge kernel reads the pairs' parts
    // itself: entries_only): no in-cluster combine. Every CTA writes its
    // unnormalized O^T (its 256 columns, the rows it holds) and its row maxima and sums as the
    // entry of its pair (entry = chunk * pairs + pair, pairs = subs * pairs per cluster) in the
    // workspace; per chunk and half a ticket counts the CTAs, and the one that takes the last
    // merges the half's columns over all the chunk's entries, in entry order (the result does not
    // depend on which pair finished last), into the chunk's slot, half 0 also the LSE; it then
    // resets the ticket. The cluster barrier split around it keeps every CTA until its peer has
    // left the tile loop (no remote store or commit reaches a CTA that has left). Its arrival
    // orders no memory: every partial-score store and commit the peer sent to this CTA was
    // waited for on this CTA's mbarriers inside the loop, and a release here cost ~0.5 us.
    cluster_arrive_relaxed();
    const int npairs_tot = subs * cluster_pairs;
    const long long entry = static_cast<long long>(chunk) * npairs_tot + pair_index;
    float* const eo = p.ws_partials + entry * rows_total * kRank;                     // [rows][512]
    float* const eml = p.ws_lse + (entry * 2 + half) * rows_total * 2;               // [rows][m, l]
    if (warp < kSoftmaxWarps) {
      const int q4 = warp & 3, h = warp >> 2;
      const float cs = p.cache_scale;  // an E4M3 cache's scale (one rounding; exact for a power of two)
      if (have) tc_fence_after();
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        float v[kRH];
        if (have) {
          tmem_ld8(tmem + tmem_lane_base(q4) + 2 * kNR + blk * kNR + kRH * h, v);
          tmem_wait_ld();
          if (kFp8)
#pragma unroll
            for (int k = 0; k < kRH; ++k) v[k] *= cs;
        } else {
#pragma unroll
          for (int k = 0; k < kRH; ++k) v[k] = 0.f;
        }
        const int col = kHalfCols * half + blk * 128 + q4 * 32 + lane;
#pragma unroll
        for (int k = 0; k < kRH; ++k)
          if (kRH * h + k < w.nrows) eo[static_cast<long long>(w.row0 + kRH * h + k) * kRank + col] = v[k];
      }
      if (tid < w.nrows) {
        eml[(w.row0 + tid) * 2] = have ? sm->mref[tid] : -INFINITY;
        eml[(w.row0 + tid) * 2 + 1] =
            have ? (sm->red[0][tid] + sm->red[1][tid]) + (sm->red[2][tid] + sm->red[3][tid]) : 0.f;
      }
    }
    __syncthreads();
    if (tid == 0) {
      // releases this CTA's entry (ordered before this thread by the barrier) with the count; the last
      // acquires the other pairs' entries before this CTA reads them. With entries_only the merge
      // kernel, a dependent launch, reads the entries after this grid has completed: no ticket.
      int last = 0;
      if (!p.entries_only) {
        uint32_t* ticket = p.ws_tickets + static_cast<long long>(chunk) * 2 + half;
        const uint32_t t = ticket_add_acq_rel(ticket);
        last = (t == static_cast<uint32_t>(npairs_tot - 1)) ? 1 : 0;
        if (last) ticket_reset(ticket);
      }
      sm->last_cluster = last;
    }
    __syncthreads();
    if (sm->last_cluster) {
      const float* const ebase = p.ws_partials + static_cast<long long>(chunk) * npairs_tot * rows_total * kRank;
      const float* const mbase = p.ws_lse + static_cast<long long>(chunk) * npairs_tot * 2 * rows_total * 2 +
                              static_cast<long long>(half) * rows_total * 2;
      const long long estride = static_cast<long long>(rows_total) * kRank;  // one entry's O
      const long long mstride = 2LL * rows_total * 2;                        // one entry's two m/l copies
      // item = 4 columns of a row (or, half 0, a row's LSE): the values, row maximum and sum of
      // up to 12 entries at once (one round trip), reduced in entry order; more entries take
      // further rounds, a larger maximum rescaling what earlier rounds summed
      const int n4 = kHalfCols / 4;
      // (single-launch decode: half 1 writes its own copy of the LSE, for its final merge)
      const int items = w.nrows * n4 + ((half == 0 || fused) ? w.nrows : 0);
      float* const lse_dst = half ? p.lse_copy : p.lse;
      for (int idx = tid; idx < items; idx += kThreads) {
        const bool is_lse = idx >= w.nrows * n4;
        const int r = is_lse ? idx - w.nrows * n4 : idx / n4;
        const int c = kHalfCols * half + (is_lse ? 0 : (idx % n4) * 4);
        const long long rowoff = static_cast<long long>(w.row0 + r);
        float M = -INFINITY, den = 0.f;
        float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int e0 = 0; e0 < npairs_tot; e0 += 12) {
          float2 ml[12];
          float4 v[12];
#pragma unroll
          for (int jj = 0; jj < 12; ++jj) {
            ml[jj] = make_float2(-INFINITY, 0.f);
            v[jj] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e0 + jj < npairs_tot) {
              ml[jj] = __ldcg(reinterpret_cast<const float2*>(mbase + (e0 + jj) * mstride + rowoff * 2));
              if (!is_lse) v[jj] = __ldcg(reinterpret_cast<const float4*>(ebase + (e0 + jj) * estride + rowoff * kRank + c));
            }
          }
          float Mr = M;
#pragma unroll
          for (int jj = 0; jj < 12; ++jj) Mr = fmaxf(Mr, ml[jj].x);
          if (Mr != -INFINITY) {
            if (M != Mr) {
              const float sc = (M == -INFINITY) ? 0.f : exp2f(M - Mr);
              den *= sc;
              num = make_float4(num.x * sc, num.y * sc, num.z * sc, num.w * sc);
            }
#pragma unroll
            for (int jj = 0; jj < 12; ++jj) {
              const float wj = (ml[jj].x == -INFINITY) ? 0.f : exp2f(ml[jj].x - Mr);
              den = fmaf(wj, ml[jj].y, den);
              num.x = fmaf(wj, v[jj].x, num.x);
              num.y = fmaf(wj, v[jj].y, num.y);
              num.z = fmaf(wj, v[jj].z, num.z);
              num.w = fmaf(wj, v[jj].w, num.w);
            }
          }
          M = Mr;
        }
        if (is_lse) {
          lse_dst[static_cast<long long>(w.slot) * rows_total + rowoff] = (M == -INFINITY) ? -INFINITY : M + log2f(den);
        } else {
          float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
          if (M != -INFINITY) o = make_float4(num.x / den, num.y / den, num.z / den, num.w / den);
          *reinterpret_cast<float4*>(p.partials + (static_cast<long long>(w.slot) * rows_total + rowoff) * kRank + c) = o;
        }
      }
      if (fused) {
        // the chunk's partial (this half) is written: count it for the request; the CTA that
        // counts the request's last chunk for this half merges the half's columns into the output
        __syncthreads();
        if (tid == 0) {
          uint32_t* ticket = p.req_tickets + static_cast<long long>(w.b) * kSliceTickets + half;
          const uint32_t t = ticket_add_acq_rel(ticket);
          const int last = (t == static_cast<uint32_t>(req_hi - req_lo - 1)) ? 1 : 0;
          if (last) ticket_reset(ticket);
          sm->last_request = last;
        }
        __syncthreads();
        if (sm->last_request)
          request_merge(p, w.b, req_lo, req_hi, kHalfCols * half, kHalfCols, half == 0, half ? p.lse_copy : p.lse,
                        tid, kThreads);
      }
    }
    cluster_wait_acquire();
    // after an abort: stores the peer issued before it left the tile loop may still be in flight
    if (!have && ntiles > 0) settle_in_flight(20000ull);
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
      tc_fence_after();
      tmem_dealloc(tmem, kTmemCols);
    }
    return;
  }
  float* ostage = reinterpret_cast<float*>(smem + kOffTile);  // [16][256]: this CTA's columns
  float* mst = ostage + kNR * kHalfCols;
  float* lst = mst + kNR;
  if (warp < kSoftmaxWarps) {
    const int q4 = warp & 3, h = warp >> 2;
    if (have) {
      tc_fence_after();
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        float v[kRH];
        tmem_ld8(tmem + tmem_lane_base(q4) + 2 * kNR + blk * kNR + kRH * h, v);
        tmem_wait_ld();
        const int d = blk * 128 + q4 * 32 + lane;
#pragma unroll
        for (int k = 0; k < kRH; ++k) ostage[(kRH * h + k) * kHalfCols + d] = kFp8 ? v[k] * p.cache_scale : v[k];
      }
    } else {
      for (int idx = tid; idx < kNR * kHalfCols; idx += kSoftmaxThreads) ostage[idx] = 0.f;
    }
    if (tid < kNR) {
      mst[tid] = have ? sm->mref[tid] : -INFINITY;
      lst[tid] = have ? (sm->red[0][tid] + sm->red[1][tid]) + (sm->red[2][tid] + sm->red[3][tid]) : 0.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  // after an abort: the remote stores the peer issued before it reached this barrier (it issues
  // none after it) may still be in flight; give them time to land before this CTA can leave
  if (!have && ntiles > 0) settle_in_flight(20000ull);
  // the cluster's result goes to the chunk's slot
  float* const dst_partials = p.partials;
  float* const dst_lse = p.lse;
  const long long dst_slot = static_cast<long long>(w.slot);
  {
    // Combine the pairs of the cluster in rank order: this CTA writes output
    // columns [rank * 512 / n, (rank + 1) * 512 / n), held by the CTAs of
    // half h = those columns / 256; rank 0 also writes the LSE.
    const int npairs = cluster_pairs;
    const int dcols = kRank / static_cast<int>(nranks);
    const int dbeg = static_cast<int>(rank) * dcols;
    const uint32_t h = static_cast<uint32_t>(dbeg / kHalfCols);
    const int n4 = dcols / 4;
    const int items = w.nrows * n4 + ((rank == 0) ? w.nrows : 0);
    for (int idx = tid; idx < items; idx += kThreads) {
      const bool is_lse = idx >= w.nrows * n4;
      const int r = is_lse ? idx - w.nrows * n4 : idx / n4;
      const int d = is_lse ? 0 : dbeg + (idx % n4) * 4;
      // every load of this item at once (one round trip), then the fixed-order reduction
      float mj[8], lj[8];
      float4 vj[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        mj[j] = -INFINITY;
        lj[j] = 0.f;
        vj[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j < npairs) {
          const uint32_t src = 2 * j + h;
          mj[j] = dsmem_ld_f32(dsmem_addr(mst + r, src));
          lj[j] = dsmem_ld_f32(dsmem_addr(lst + r, src));
          if (!is_lse) vj[j] = dsmem_ld_f32x4(dsmem_addr(ostage + r * kHalfCols + (d - kHalfCols * h), src));
        }
      }
      float M = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) M = fmaxf(M, mj[j]);
      float den = 0.f;
      float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
      if (M != -INFINITY) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float wj = (mj[j] == -INFINITY) ? 0.f : exp2f(mj[j] - M);
          den = fmaf(wj, lj[j], den);
          num.x = fmaf(wj, vj[j].x, num.x);
          num.y = fmaf(wj, vj[j].y, num.y);
          num.z = fmaf(wj, vj[j].z, num.z);
          num.w = fmaf(wj, vj[j].w, num.w);
        }
      }
      if (is_lse) {
        dst_lse[dst_slot * rows_total + w.row0 + r] = (M == -INFINITY) ? -INFINITY : M + log2f(den);
      } else {
        float4 out = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) out = make_float4(num.x / den, num.y / den, num.z / den, num.w / den);
        const long long base = (dst_slot * rows_total + w.row0 + r) * kRank + d;
        *reinterpret_cast<float4*>(dst_partials + base) = out;
      }
    }
  }
  cluster_sync();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (fused) {
    // Single-launch decode: the cluster's chunk partial is complete (every rank wrote its column
    // slice, rank 0 the LSE, all before the barrier above). Per request and slice a ticket counts
    // the chunks; the CTA that counts the last one merges that slice of all the request's
    // partials into the output (rank 0's slice also the merged LSE).
    const int dcols = kRank / static_cast<int>(nranks);
    if (tid == 0) {
      // the cluster's slices and rank 0's LSE are ordered before this thread by the cluster barrier;
      // the acquire-release add releases them at device scope with the count (and, for the last,
      // acquires the other clusters' partials before this CTA's threads read them after the
      // barrier below)
      uint32_t* ticket = p.req_tickets + static_cast<long long>(w.b) * kSliceTickets + rank;
      const uint32_t t = ticket_add_acq_rel(ticket);
      const int last = (t == static_cast<uint32_t>(req_hi - req_lo - 1)) ? 1 : 0;
      if (last) ticket_reset(ticket);
      sm->last_request = last;
    }
    __syncthreads();
    if (sm->last_request)
      request_merge(p, w.b, req_lo, req_hi, static_cast<int>(rank) * dcols, dcols, rank == 0, p.lse, tid, kThreads);
  }
}

template <bool kFp8, bool kBf16>
cudaError_t prepare(int cluster) {
  static bool smem_set = false, np_set = false;
  const void* fn = reinterpret_cast<const void*>(&mla_partial_tc128_kernel<kFp8, kBf16>);
  cudaError_t e = cudaSuccess;
  if (!smem_set) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    smem_set = true;
  }
  if (cluster > 8 && !np_set) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    np_set = true;
  }
  return e;
}

}  // namespace

bool tc128_supports(int total_rows, bool, int cluster) {
  return total_rows <= kNR && cluster >= 2 && cluster <= 16 && (cluster & (cluster - 1)) == 0;
}

cudaError_t launch_partial_tc128(const CUtensorMap& tm_pages, const CUtensorMap& tm_kpe_half, const PartialParams& p,
                                 int num_chunks, int cluster, bool bf16, cudaStream_t stream) {
  if (p.fp8 && bf16) return cudaErrorInvalidValue;  // E4M3 caches go with fp16 queries
  cudaError_t e = p.fp8 ? prepare<true, false>(cluster)
                  : bf16 ? prepare<false, true>(cluster) : prepare<false, false>(cluster);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster, num_chunks * (p.subs > 1 ? p.subs : 1), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (p.fp8) return cudaLaunchKernelEx(&cfg, mla_partial_tc128_kernel<true, false>, tm_pages, tm_kpe_half, p);
  return bf16 ? cudaLaunchKernelEx(&cfg, mla_partial_tc128_kernel<false, true>, tm_pages, tm_kpe_half, p)
              : cudaLaunchKernelEx(&cfg, mla_partial_tc128_kernel<false, false>, tm_pages, tm_kpe_half, p);
}

int tc128_max_active_clusters(int cluster) {
  // every instance takes the same threads, shared memory and (at most) registers
  if (prepare<false, false>(cluster) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(&mla_partial_tc128_kernel<false, false>), &cfg) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t tc128_read_clear_error(uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_device_error, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(uint32_t));
}

}  // namespace mla
