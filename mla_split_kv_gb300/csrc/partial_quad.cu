// Tensor-core partial-decode kernel for CTAs of 16 query rows (fp16) working
// in quads, sm_103a.
//
// The operation is the one of the other partial kernels ("feat(core):
// matrix-absorbed MLA decode over a compressed-latent KV cache", *What
// changed*: SDPA(q_absorbed, ckv, ckv, scale, mask = scale * q_pe @ kpe^T),
// each chunk yielding a normalized partial and its log2 LSE).
//
// 16 query rows are too few for the tensor core's M side, so tokens and
// latent columns go on M=128 and the rows on N=16. A 128-token tile of the
// whole latent (144 KB) cannot stay in one SM from the score product to the PV
// product while the next tiles load, so the four CTAs of a quad (cluster ranks
// 4g .. 4g+3, quad rank q) share each tile and split it two ways:
//
//   scores, split by columns. CTA q loads ckv columns [128 q, 128 q + 128) and
//   kpe columns [16 q, 16 q + 16) of the 128 tokens (36 KB) and computes the
//   partial scores over them, S_q^T[tok, row] (M=128 tokens, K=144, N=16). A
//   reduce-scatter through distributed shared memory gives CTA q the complete
//   scores of its own 32 tokens [32 q, 32 q + 32): warp w of every CTA holds
//   TMEM lanes 32w.. (tokens 32w..), so it sends them to CTA w, which adds the
//   four parts in rank order.
//
//   values, split by tokens. CTA q runs the softmax of its 32 tokens with its
//   own running max and sum and accumulates O^T[d, row] over all 512 columns
//   for them (four M=128 column blocks, K=32). The other CTAs' columns of
//   those tokens are 8 KB runs of their tile slots (8-token row groups 4q ..
//   4q+3), so each CTA bulk-copies them to their owners as soon as a tile has
//   landed, off the softmax's path.
//
// Every CTA ends with its own (max, sum, O) over a quarter of the tokens; the
// cluster combines them at the end, in rank order, like partitions. Per CTA and
// tile that is 9 score MMAs and 8 PV MMAs, the softmax of 32 x 16 scores, and
// 36 KB of tile slot, so four slots fit: tiles i+1 .. i+3 load while tile i is
// computed.
//
// The ckv columns arrive as one 4D TMA box per page (64 columns x 8 rows x 2
// column blocks x page/8 row groups): row group g, block c at 2048 g + 1024 c,
// swizzled [8 x 64] atoms. Score MMAs read it K-major (8-row groups 2 KB
// apart), PV MMAs MN-major (the two 64-column halves of an M=128 block 1 KB
// apart, 8-token groups 2 KB apart). The kpe columns are a [tokens x 32 B] box
// with the 32-byte swizzle (one K=16 step).
//
// Warp roles (256 threads, two warps per scheduler so that each may hold 255
// registers): warps 0-3 softmax (thread = token lane of S^T; warp q, whose
// lanes hold this CTA's own tokens, runs their softmax; the others send their
// lanes' partial scores to their owners and rescale their lanes of O^T when
// the owner asks), warp 4 TMEM owner and MMA issuer (score or PV product,
// whichever is ready first), warp 5 copies to the other CTAs, warps 6-7 page
// producers (warp 6+k loads pages k, k+2, ... of each tile).
#include "device_common.cuh"

namespace mla {

namespace {

constexpr int kT = 128;                              // tokens per tile
constexpr int kNR = 16;                              // query rows per CTA
constexpr int kQuad = 4;                             // CTAs sharing a tile
constexpr int kQCols = kRank / kQuad;                // 128 ckv columns of the score product per CTA
constexpr int kQBoxes = kQCols / kBoxCols;           // 2 column blocks of 64
constexpr int kQKpe = kRope / kQuad;                 // 16 kpe columns per CTA
constexpr int kQTok = kT / kQuad;                    // 32 tokens of the PV product per CTA
constexpr int kGroupBytes = 8 * kQCols * 2;          // 2 KB: one 8-token row group of the two blocks
constexpr int kCkvBytes = kT * kQCols * 2;           // 32 KB
constexpr int kKpeBytes = kT * kQKpe * 2;            // 4 KB: [128 tokens x 32 B], 32-byte swizzle
constexpr int kTileSlot = kCkvBytes + kKpeBytes;     // 36 KB
constexpr int kSlots = 4;
constexpr int kVChunk = kQTok * kQCols * 2;          // 8 KB: one CTA's columns of a quarter's tokens
constexpr int kPrefetch = kSlots;                    // L2 prefetch distance in tiles
constexpr int kSoftmaxThreads = 128;
constexpr int kPageWarps = 2;                        // producer warps
constexpr int kThreads = (6 + kPageWarps) * 32;      // 256: two warps per scheduler
constexpr float kRescaleTau = 8.0f;

constexpr uint32_t kOffTile = 0;                             // 4 tile slots
constexpr uint32_t kOffQ = kSlots * kTileSlot;               // 144 KB: Q^T, 3 chunks
constexpr uint32_t kQChunk = kNR * 128;                      // [16 x 64] fp16, swizzled: 2 KB
constexpr uint32_t kOffV = kOffQ + 3 * kQChunk;              // 150 KB: other CTAs' columns, 2 buffers
constexpr uint32_t kVBuf = (kQuad - 1) * kVChunk;            // 24 KB
constexpr uint32_t kOffRS = kOffV + 2 * kVBuf;               // 198 KB: other CTAs' partial scores, 2 buffers
constexpr uint32_t kRSPart = kQTok * kNR * 4;                // [32 tokens][16 rows] fp32: 2 KB
constexpr uint32_t kRSBuf = (kQuad - 1) * kRSPart;           // 6 KB
constexpr uint32_t kOffP = kOffRS + 2 * kRSBuf;              // 210 KB: P^T, 2 buffers
constexpr uint32_t kPBuf = kNR * 128;                        // [16 rows x 64-token atom], 32 tokens used
constexpr uint32_t kOffSmall = kOffP + 2 * kPBuf;            // 214 KB
constexpr uint32_t kSmem = kOffSmall + 1024 + 1024;          // + alignment slack
constexpr uint32_t kTmemCols = 128;                          // S^T 2 x 16 + O^T 4 x 16
static_assert(kSmem <= 232448, "shared memory per CTA");
static_assert(kNR * kRank * 4 + 2 * kNR * 4 <= kSlots * kTileSlot, "epilogue staging fits the tile slots");
static_assert(kOffV % 1024 == 0 && kOffP % 1024 == 0 && kTileSlot % 1024 == 0, "swizzled operands on 1 KB");

struct Small {
  uint64_t full[kSlots], empty[kSlots];
  uint64_t sfull[2], sfree[2];
  uint64_t rsfull[2];          // the other CTAs' partial scores of this CTA's tokens have landed
  uint64_t rsfree[kQuad][2];   // [receiver]: that CTA has read its buffer (remote arrival)
  uint64_t vfull[2];           // the other CTAs' columns of this CTA's tokens have landed
  uint64_t vfree[kQuad][2];    // [receiver]: that CTA's PV product read its buffer (remote commit)
  uint64_t pfull[2], pvdone[2];
  uint64_t req[4];             // the owner warp's decision for tile j (slot j & 3): flag[j & 3]
  uint64_t rescaled;           // the other softmax warps rescaled their lanes of O^T
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t last_cluster;  // this cluster took the chunk's last ticket
  int32_t any_pv;
  int32_t flag[4];             // 1: rescale O^T by alpha[j & 3] before PV(j)
  float alpha[4][kNR];
};
static_assert(sizeof(Small) <= 1024, "small smem region");

__device__ __forceinline__ uint32_t tmem_lane_base(int warp) { return static_cast<uint32_t>(32 * (warp & 3)) << 16; }
// Buffer index of sender `from` in receiver `to`'s buffers (the three other quad ranks, ascending).
__device__ __forceinline__ int sender_index(int from, int to) { return from < to ? from : from - 1; }

__global__ void __launch_bounds__(kThreads, 1)
    mla_partial_quad_kernel(const __grid_constant__ CUtensorMap tm_pages, const __grid_constant__ CUtensorMap tm_kpe,
                            const PartialParams p) {
  extern __shared__ uint8_t smem_raw[];
  pdl_launch_dependents();  // the merge of these partials may be scheduled now; it waits for this grid
  uint8_t* smem = align1024(smem_raw);
  uint8_t* qs = smem + kOffQ;
  uint8_t* ps = smem + kOffP;
  uint8_t* vs = smem + kOffV;
  float* rs = reinterpret_cast<float*>(smem + kOffRS);
  Small* sm = reinterpret_cast<Small*>(smem + kOffSmall);
  volatile int32_t* abort_flag = &sm->abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank(), nranks = cluster_nctarank();
  const int qr = static_cast<int>(rank & 3u);            // quad rank: column quarter, token quarter
  const uint32_t quad_base = rank & ~3u;                 // cluster rank of quad rank 0
  // a chunk may be spread over `subs` clusters (grid.y = chunk * subs + sub); its tiles are
  // split over all their quads
  const int subs = (p.subs > 1) ? p.subs : 1;
  const int chunk = static_cast<int>(blockIdx.y) / subs, sub = static_cast<int>(blockIdx.y) % subs;
  const int cluster_quads = static_cast<int>(nranks >> 2);
  const CtaWork w =
      cta_work(p, kNR, kT, sub * cluster_quads + static_cast<int>(rank >> 2), subs * cluster_quads, chunk);
  const int ntiles = (w.sub1 - w.sub0 + kT - 1) / kT;
  const int rows_total = p.q_len * p.H;
  // valid tokens of this CTA's quarter in tile i
  auto quarter_valid = [&](int i) -> int {
    const int nv = min(kT, w.sub1 - (w.sub0 + i * kT)) - kQTok * qr;
    return nv < 0 ? 0 : (nv > kQTok ? kQTok : nv);
  };

  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&sm->full[s], kPageWarps);  // one expect_tx arrival per producer warp
      // this CTA's PV product + the three other CTAs, once their copies of the slot have landed
      mbar_init(&sm->empty[s], 1 + (kQuad - 1));
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm->sfull[t], 1);
      mbar_init(&sm->sfree[t], 4);
      mbar_init(&sm->rsfull[t], 1);  // local expect_tx arrival + the other CTAs' st.async bytes
      mbar_init(&sm->vfull[t], 1);   // local expect_tx arrival + the other CTAs' bulk copies
      mbar_init(&sm->pfull[t], 1);
      mbar_init(&sm->pvdone[t], 1);
      for (int k = 0; k < kQuad; ++k) {
        mbar_init(&sm->rsfree[k][t], 1);
        mbar_init(&sm->vfree[k][t], 1);
      }
    }
    for (int k = 0; k < 4; ++k) mbar_init(&sm->req[k], 1);
    mbar_init(&sm->rescaled, kQuad - 1);
    mbar_init(&sm->drain, 1);
    for (int t = 0; t < 2 && t < ntiles; ++t) {  // tiles 0 and 1
      mbar_arrive_expect_tx(&sm->rsfull[t], kRSBuf);
      mbar_arrive_expect_tx(&sm->vfull[t], kVBuf);
    }
    sm->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(&sm->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive_release();  // the other CTAs touch this CTA's barriers only after this cluster phase
  const uint32_t tmem = sm->tmem_base;
  bool any_pv = false;  // softmax warps: some tile had tokens in this CTA's quarter
  // owner warp of the softmax: reference max and running sum of each row over this CTA's tokens
  float mr[kNR], lsum[kNR];
#pragma unroll
  for (int r = 0; r < kNR; ++r) {
    mr[r] = -INFINITY;
    lsum[r] = 0.f;
  }

  if (warp >= 6) {
    // ------------------------------------------------------------------ producers
    const int k0 = warp - 6;  // this warp loads pages k0, k0 + kPageWarps, ... of each tile
    const uint64_t pol = l2_policy_evict_first();
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
    int issued = -1;
    for (int i = 0; i < ntiles; ++i) {
      const int s = i % kSlots;
      if (i >= kSlots) {  // tile i - kSlots released the slot
        int ok = 1;
        if (lane == 0) {
          ok = mbar_wait(&sm->empty[s], ((i / kSlots) - 1) & 1, p.timeout_ns) && !*abort_flag;
          if (!ok) *abort_flag = 1;
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
      int pg0, npg;
      tile_pages(i, &pg0, &npg);
      const int mine = (npg > k0) ? (npg - k0 + kPageWarps - 1) / kPageWarps : 0;
      uint8_t* slot = smem + kOffTile + s * kTileSlot;
      if (lane == 0)
        mbar_arrive_expect_tx(&sm->full[s], static_cast<uint32_t>(mine * p.bs * (kQCols + kQKpe) * 2));
      for (int m = 0; m < mine; ++m) {
        const int j = k0 + m * kPageWarps;  // page of the tile
        const int pid = page_of(pg0 + j);
        if (lane == 0) {
          tma_load_4d(slot + j * p.bs * (kQCols * 2), &tm_pages, 0, 0, kQBoxes * qr, pid * (p.bs / 8), &sm->full[s],
                      pol);
          tma_load_2d(slot + kCkvBytes + j * p.bs * (kQKpe * 2), &tm_kpe, kQKpe * qr, pid * p.bs, &sm->full[s], pol);
        }
      }
      issued = i;
      if (i + kPrefetch < ntiles) {  // pages of tile i + kPrefetch into L2: a quarter of them per CTA
        int qg0, qn;
        tile_pages(i + kPrefetch, &qg0, &qn);
        for (int j = k0; j < qn; j += kPageWarps) {
          if ((j & 3) != qr) continue;
          const int pid = page_of(qg0 + j);
          if (lane == 0 && pid >= 0) {
            const long long row = static_cast<long long>(pid) * p.bs;
            bulk_prefetch_l2(p.ckv + row * (kRank * 2), static_cast<uint32_t>(p.bs * kRank * 2));
            bulk_prefetch_l2(p.kpe + row * (kRope * 2), static_cast<uint32_t>(p.bs * kRope * 2));
          }
        }
      }
    }
    // after an abort, let this warp's last loads land before shared memory is released
    if (lane == 0 && *abort_flag && issued >= 0)
      mbar_wait(&sm->full[issued % kSlots], (issued / kSlots) & 1, kDrainTimeoutNs);
    cluster_wait_acquire();
  } else if (warp == 5) {
    // ------------------------------------------------------------------ copies to the other CTAs
    // Tile i's rows of quad rank k (row groups 4k .. 4k+3 of the slot, this CTA's 128 columns)
    // go to CTA k's column buffer once the tile has landed here and CTA k's PV product of
    // tile i-2 has released that buffer.
    cluster_wait_acquire();
    if (lane == 0) {
      uint64_t tmo = p.timeout_ns;
      bool ok = true;
      int copied = -1;
      for (int i = 0; i < ntiles && ok; ++i) {
        const int s = i % kSlots, t = i & 1;
        ok = mbar_wait(&sm->full[s], (i / kSlots) & 1, tmo) && !*abort_flag;
        const uint8_t* slot = smem + kOffTile + s * kTileSlot;
        for (int k = 1; k < kQuad && ok; ++k) {
          const int to = (qr + k) & 3;
          if (i >= 2) ok = mbar_wait_cluster(&sm->vfree[to][t], ((i >> 1) - 1) & 1, tmo) && !*abort_flag;
          if (!ok) break;
          const uint32_t dst_rank = quad_base + static_cast<uint32_t>(to);
          const uint32_t dst = dsmem_addr(vs + t * kVBuf + sender_index(qr, to) * kVChunk, dst_rank);
          dsmem_bulk_copy(dst, slot + (4 * to) * kGroupBytes, kVChunk, dsmem_addr(&sm->vfull[t], dst_rank));
        }
        if (ok) copied = i;
      }
      if (!ok) *abort_flag = 1;
      // the receivers' last two PV products have released their buffers (their remote commits
      // land here) before this CTA may exit
      const uint64_t tmo_end = ok ? tmo : kDrainTimeoutNs / 8;
      for (int i = (copied >= 1 ? copied - 1 : 0); i <= copied; ++i)
        for (int k = 1; k < kQuad; ++k)
          if (!mbar_wait_cluster(&sm->vfree[(qr + k) & 3][i & 1], (i >> 1) & 1, tmo_end)) *abort_flag = 1;
    }
    __syncwarp();
  } else if (warp == 4) {
    // ------------------------------------------------------------------ MMA issuer
    const uint32_t idesc_s = idesc_f16_f32(128, kNR, false, false, false);
    const uint32_t idesc_o = idesc_f16_f32(128, kNR, false, true, false);
    const Desc2 qd = desc2(smem_desc_sw128(smem_u32(qs), 16, 1024));
    const Desc2 pd = desc2(smem_desc_sw128(smem_u32(ps), 16, 1024));
    const uint32_t tile_base = smem_u32(smem + kOffTile);
    const uint16_t peer_mask = static_cast<uint16_t>((0xFu << quad_base) & ~(1u << rank));
    uint64_t tmo = p.timeout_ns;
    asm volatile("" : "+l"(tmo));
    // score product of tile i into S buffer i&1: this CTA's two ckv column blocks, then its kpe step
    auto score = [&](int i) {
      const int t = i & 1, s = i % kSlots;
      if (lane == 0) {
        tc_fence_after();
        const uint32_t slot = tile_base + s * kTileSlot;
        const Desc2 ad = desc2(smem_desc_sw128(slot, 16, kGroupBytes));
        const uint32_t d = tmem + t * kNR;
#pragma unroll
        for (int c = 0; c < kQBoxes; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ss(d, ad, (c * 1024 + kk * 32) >> 4, qd, (c * kQChunk + kk * 32) >> 4, idesc_s,
                    (c == 0 && kk == 0) ? 0u : 1u);
        umma_ss(d, desc2(smem_desc_sw32(slot + kCkvBytes, 256)), 0, qd, (kQBoxes * kQChunk) / 16 + qr * 2, idesc_s, 1u);
        umma_commit(&sm->sfull[t]);
      }
      __syncwarp();
    };
    // rows [nq, nend) of this CTA's quarter in a column block (own slot or a copy): zeroed so the
    // PV operand stays finite (their probabilities are 0, but rows past the context may hold anything)
    auto zero_rows = [&](uint8_t* blk, int nq, int nend) {
      for (int x = lane; x < (nend - nq) * kQBoxes * 8; x += 32) {
        const int rc = x >> 3, tok = nq + rc / kQBoxes, c = rc % kQBoxes;
        *reinterpret_cast<uint4*>(blk + (tok >> 3) * kGroupBytes + c * 1024 + (tok & 7) * 128 + (x & 7) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
    };
    bool o_started = false;
    // PV product of tile i: O^T block c (columns [128 c, 128 c + 128)) += ckv^T . P^T over this
    // CTA's tokens; block qr from the own slot, the others from the copies
    auto pv = [&](int i) {
      const int t = i & 1, s = i % kSlots;
      const int nq = quarter_valid(i);
      const int ksteps = (nq + 15) >> 4;
      if (lane == 0) {
        // the copies have landed: their senders' slots are free as far as this CTA goes
        for (int k = 1; k < kQuad; ++k)
          mbar_remote_arrive_relaxed(dsmem_addr(&sm->empty[s], quad_base + ((qr + k) & 3)));
      }
      uint8_t* own = smem + kOffTile + s * kTileSlot + (4 * qr) * kGroupBytes;
      if (nq > 0 && nq < (ksteps << 4)) {
        zero_rows(own, nq, ksteps << 4);
        for (int k = 0; k < kQuad - 1; ++k) zero_rows(vs + t * kVBuf + k * kVChunk, nq, ksteps << 4);
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        // the copies of tile i+2 may come once this commit releases the buffer
        if (i + 2 < ntiles) mbar_arrive_expect_tx(&sm->vfull[t], kVBuf);
        tc_fence_after();
        const Desc2 pb = desc2_add(pd, t * kPBuf);
        const uint32_t acc0 = o_started ? 1u : 0u;
#pragma unroll
        for (int c = 0; c < kQuad; ++c) {
          const uint32_t base = (c == qr) ? smem_u32(own) : smem_u32(vs + t * kVBuf + sender_index(c, qr) * kVChunk);
          const Desc2 a0 = desc2(smem_desc_sw128(base, 1024, kGroupBytes));
          const uint32_t d = tmem + 2 * kNR + c * kNR;
          if (ksteps == 2) {
            umma_ss(d, a0, 0, pb, 0, idesc_o, acc0);
            umma_ss(d, a0, (2 * kGroupBytes) >> 4, pb, 32 >> 4, idesc_o, 1u);
          } else if (ksteps == 1) {
            umma_ss(d, a0, 0, pb, 0, idesc_o, acc0);
          }
        }
        umma_commit(&sm->pvdone[t]);
        umma_commit(&sm->empty[s]);
        umma_commit_multicast(&sm->vfree[qr][t], peer_mask);
      }
      if (ksteps > 0) o_started = true;
      __syncwarp();
    };
    named_bar_sync(2, 32 * 5);  // Q^T staged by the softmax warps
    cluster_wait_acquire();
    // Whichever product is ready first, each kind in tile order: S(ns) once tile ns has landed
    // and the softmax has read S buffer ns & 1 (tile ns-2); PV(np) once P of tile np is written
    // and the other CTAs' copies of tile np have landed.
    int ns = 0, np = 0;
    bool alive = true;
    uint64_t t0 = 0;
    while (np < ntiles && alive) {
      int pick = 0;  // 1: S, 2: PV, -1: abort
      if (lane == 0) {
        if (ns < ntiles && (ns < 2 || mbar_test(&sm->sfree[ns & 1], ((ns >> 1) - 1) & 1)) &&
            mbar_test(&sm->full[ns % kSlots], (ns / kSlots) & 1))
          pick = 1;
        else if (np < ns && mbar_test(&sm->pfull[np & 1], (np >> 1) & 1) &&
                 mbar_test(&sm->vfull[np & 1], (np >> 1) & 1))
          pick = 2;
        else if (*abort_flag)
          pick = -1;
        if (pick == 2) mbar_wait_cluster(&sm->vfull[np & 1], (np >> 1) & 1, tmo);  // cluster-scope acquire
      }
      pick = __shfl_sync(0xffffffffu, pick, 0);
      if (pick == 1) {
        score(ns++);
      } else if (pick == 2) {
        pv(np++);
      } else if (pick < 0) {
        alive = false;
      } else {
        const uint64_t now = globaltimer_ns();
        if (t0 == 0) t0 = now;
        if (now - t0 > tmo) {
          if (lane == 0) {
            flag_error(MLA_DEVERR_TIMEOUT);
            *abort_flag = 1;
          }
          alive = false;
        }
        continue;
      }
      t0 = 0;
    }
    if (!alive && lane == 0) *abort_flag = 1;
    if (lane == 0) {  // every MMA issued so far has completed before TMEM is read or freed
      umma_commit(&sm->drain);
      mbar_wait(&sm->drain, 0, kDrainTimeoutNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax (warps 0-3)
    float scale_log2 = p.scale_log2;
    uint64_t tmo = p.timeout_ns;
    asm volatile("" : "+f"(scale_log2), "+l"(tmo));
    // Q^T: this CTA's 128 latent columns, then the 64 kpe columns; 16 rows, K-major, 3 swizzled chunks
    for (int idx = tid; idx < kNR * 3 * 8; idx += kSoftmaxThreads) {
      const int r = idx / (3 * 8), k = (idx % (3 * 8)) * 8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (r < w.nrows) {
        const long long row = static_cast<long long>(w.b) * rows_total + w.row0 + r;
        v = (k < kQCols) ? *reinterpret_cast<const uint4*>(p.q_abs + row * kRank + kQCols * qr + k)
                         : *reinterpret_cast<const uint4*>(p.q_pe + row * kRope + (k - kQCols));
      }
      *reinterpret_cast<uint4*>(qs + (k / kBoxCols) * kQChunk + sw128_offset(r, k % kBoxCols)) = v;
    }
    fence_proxy_async_smem();
    named_bar_arrive(2, 32 * 5);
    cluster_wait_acquire();  // the other CTAs' barriers are initialised

    const bool owner = (warp == qr);  // this warp's TMEM lanes are this CTA's own tokens
    const uint32_t xsw = static_cast<uint32_t>((lane >> 1) & 3);
    // A(i): load tile i's partial scores of this warp's 32 tokens; a non-owner sends them to the
    // CTA that owns those tokens (4 float4 chunks of row `lane`, chunk c at position
    // c ^ ((lane >> 1) & 3): conflict-free 16-byte reads), the owner keeps them.
    auto load_scores = [&](int i, float* x) -> bool {
      const int t = i & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&sm->sfull[t], (i >> 1) & 1, tmo);
      if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
      tc_fence_after();
      tmem_ld16(tmem + tmem_lane_base(warp) + t * kNR, x);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->sfree[t]);
      if (!owner) {
        const uint32_t to_rank = quad_base + static_cast<uint32_t>(warp);
        // the owner has read this buffer's previous use (tile i-2)
        if (i >= 2) ok = mbar_wait_cluster(&sm->rsfree[warp][t], ((i >> 1) - 1) & 1, tmo);
        if (!__all_sync(0xffffffffu, ok)) return false;
        const uint32_t dst = dsmem_addr(rs, to_rank) + t * kRSBuf + sender_index(qr, warp) * kRSPart + lane * 64;
        const uint32_t rbar = dsmem_addr(&sm->rsfull[t], to_rank);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          dsmem_st_async_f32x4(dst + ((c ^ xsw) << 4), make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]),
                               rbar);
      }
      return true;
    };
    // rescale of O^T requested by the owner for tile j (slot j & 3): this warp's TMEM lanes,
    // once PV(j-1) is complete
    auto rescale_o = [&](int j) -> bool {
      if (j >= 1) {
        int ok = 1;
        if (lane == 0) ok = mbar_wait(&sm->pvdone[(j - 1) & 1], ((j - 1) >> 1) & 1, tmo);
        if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
        tc_fence_after();
        const float* a = sm->alpha[j & 3];
#pragma unroll
        for (int c = 0; c < kQuad; ++c) {
          float v[16];
          const uint32_t ta = tmem + tmem_lane_base(warp) + 2 * kNR + c * kNR;
          tmem_ld16(ta, v);
          tmem_wait_ld();
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) v[jj] *= a[jj];
          tmem_st16(ta, v);
        }
        tmem_wait_st();
        tc_fence_before();
      }
      return true;
    };
    bool ok_all = true;
    if (!owner) {
      // senders: A(i) for every tile, then serve the owner's request for tile i-1
      for (int i = 0; i <= ntiles && ok_all; ++i) {
        float x[kNR];
        if (i < ntiles) ok_all = load_scores(i, x);
        if (!ok_all || i == 0) continue;
        const int j = i - 1;
        int ok = 1;
        if (lane == 0) ok = mbar_wait(&sm->req[j & 3], (j >> 2) & 1, tmo);
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          ok_all = false;
          break;
        }
        if (sm->flag[j & 3] != 0) {
          ok_all = rescale_o(j);
          __syncwarp();
          if (ok_all && lane == 0) mbar_arrive(&sm->rescaled);
        }
      }
      // every owner has read this CTA's partial scores of the last two tiles (the senders'
      // barriers see no arrival after this CTA has left)
      for (int i = (ntiles >= 2 ? ntiles - 2 : 0); i < ntiles && ok_all; ++i) {
        int ok = mbar_wait_cluster(&sm->rsfree[warp][i & 1], (i >> 1) & 1, tmo);
        ok_all = __all_sync(0xffffffffu, ok);
      }
    } else {
      const int causal_floor = p.causal ? w.L - p.q_len + w.row0 / p.H : 0x7fffffff;
      float xown[kNR], xnext[kNR];
      int nrescale = 0;
      if (ntiles > 0) ok_all = load_scores(0, xown);
      for (int j = 0; j < ntiles && ok_all; ++j) {
        const int t = j & 1;
        // A(j+1) first when its scores are ready (it frees their S buffer sooner)
        bool next_done = false;
        if (j + 1 < ntiles) {
          int ready = 0;
          if (lane == 0) ready = mbar_test(&sm->sfull[(j + 1) & 1], ((j + 1) >> 1) & 1);
          if (__shfl_sync(0xffffffffu, ready, 0)) {
            ok_all = load_scores(j + 1, xnext);
            next_done = true;
          }
        }
        // ---- B(j): complete the scores of this CTA's 32 tokens, softmax, P
        int ok = ok_all ? mbar_wait_cluster(&sm->rsfull[t], (j >> 1) & 1, tmo) : 0;
        if (!__all_sync(0xffffffffu, ok)) {
          ok_all = false;
          break;
        }
        float sc[kNR];
        {
          // the four parts in rank order (the other ranks' parts ascending in the buffer; the own
          // part takes rank qr's place): the same sum whichever CTA owns the tokens
          const float4* xb = reinterpret_cast<const float4*>(rs + t * (kRSBuf / 4) + lane * 16);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float4 y0 = xb[0 * (kRSPart / 16) + (c ^ xsw)];
            const float4 y1 = xb[1 * (kRSPart / 16) + (c ^ xsw)];
            const float4 y2 = xb[2 * (kRSPart / 16) + (c ^ xsw)];
            const float4 o = make_float4(xown[4 * c], xown[4 * c + 1], xown[4 * c + 2], xown[4 * c + 3]);
            const float4 a = (qr == 0) ? o : y0;
            const float4 b = (qr == 0) ? y0 : ((qr == 1) ? o : y1);
            const float4 d = (qr <= 1) ? y1 : ((qr == 2) ? o : y2);
            const float4 e = (qr == 3) ? o : y2;
            sc[4 * c] = ((a.x + b.x) + d.x) + e.x;
            sc[4 * c + 1] = ((a.y + b.y) + d.y) + e.y;
            sc[4 * c + 2] = ((a.z + b.z) + d.z) + e.z;
            sc[4 * c + 3] = ((a.w + b.w) + d.w) + e.w;
          }
        }
        __syncwarp();
        if (lane == 0) {
          // the buffer is read: expect tile j+2 in it, then tell the senders it is free
          if (j + 2 < ntiles) mbar_arrive_expect_tx(&sm->rsfull[t], kRSBuf);
          for (int k = 1; k < kQuad; ++k)
            mbar_remote_arrive_relaxed(dsmem_addr(&sm->rsfree[qr][t], quad_base + ((qr + k) & 3)));
        }
        const int nq = quarter_valid(j);
        if (nq > 0) any_pv = true;
        const int tok0 = w.sub0 + j * kT + kQTok * qr;
        if (__builtin_expect(nq < kQTok || tok0 + kQTok - 1 > causal_floor || w.nrows < kNR, 0)) {
#pragma unroll
          for (int r = 0; r < kNR; ++r) {
            bool vis = (lane < nq) && (r < w.nrows);
            if (p.causal) vis = vis && (tok0 + lane <= w.L - p.q_len + (w.row0 + r) / p.H);
            sc[r] = vis ? sc[r] * scale_log2 : -INFINITY;
          }
        } else {
#pragma unroll
          for (int r = 0; r < kNR; ++r) sc[r] *= scale_log2;
        }
        bool need = false;
#pragma unroll
        for (int r = 0; r < kNR; ++r) need |= sc[r] > mr[r] + kRescaleTau;
        need = __any_sync(0xffffffffu, need);
        if (__builtin_expect(need, 0)) {
          // rare path: move the reference max; every warp rescales its TMEM lanes of O^T
#pragma unroll
          for (int r = 0; r < kNR; ++r) {
            float v = sc[r];
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
            const float mnew = fmaxf(mr[r], v);
            const float a = (mnew == -INFINITY) ? 1.f : exp2f(mr[r] - mnew);
            mr[r] = mnew;
            lsum[r] *= a;
            if (lane == 0) sm->alpha[j & 3][r] = a;
          }
          __syncwarp();
          if (lane == 0) {
            sm->flag[j & 3] = 1;
            mbar_arrive(&sm->req[j & 3]);
          }
          ok_all = rescale_o(j);
          int ok2 = 1;
          if (lane == 0) ok2 = mbar_wait(&sm->rescaled, nrescale & 1, tmo);
          ++nrescale;
          if (!__shfl_sync(0xffffffffu, ok2, 0) || !ok_all) {
            ok_all = false;
            break;
          }
          tc_fence_after();
        } else if (lane == 0) {
          sm->flag[j & 3] = 0;
          mbar_arrive(&sm->req[j & 3]);
        }
        if (j >= 2) {  // P^T buffer t was last read by PV(j-2)
          int ok3 = 1;
          if (lane == 0) ok3 = mbar_wait(&sm->pvdone[t], ((j >> 1) - 1) & 1, tmo);
          if (!__shfl_sync(0xffffffffu, ok3, 0)) {
            ok_all = false;
            break;
          }
        }
        // probabilities -> P^T (fp16, K-major, 32 tokens of a swizzled 64-token atom) and row sums
        uint8_t* pb = ps + t * kPBuf;
#pragma unroll
        for (int r = 0; r < kNR; ++r) {
          // masked scores (-inf) give 0; a row with no visible token yet subtracts a finite stand-in
          const float pr = fast_exp2(sc[r] - ((mr[r] == -INFINITY) ? 0.f : mr[r]));
          const uint16_t hv = f2h<false>(pr);
          lsum[r] += h2f<false>(hv);
          *reinterpret_cast<uint16_t*>(pb + sw128_offset(r, lane)) = hv;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->pfull[t]);
        if (j + 1 < ntiles) {
          if (!next_done) ok_all = load_scores(j + 1, xnext);
#pragma unroll
          for (int r = 0; r < kNR; ++r) xown[r] = xnext[r];
        }
      }
      if (ok_all && ntiles > 0) {
        int ok = 1;
        if (lane == 0) ok = mbar_wait(&sm->pvdone[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, tmo);
        ok_all = __shfl_sync(0xffffffffu, ok, 0) != 0;
      }
    }
    if (!ok_all && lane == 0) *abort_flag = 1;
    if (owner && lane == 0) sm->any_pv = any_pv ? 1 : 0;
    named_bar_sync(1, kSoftmaxThreads);
    any_pv = sm->any_pv != 0;
  }
  __syncthreads();  // all roles done: the tile slots are free for staging
  const bool have = !*abort_flag;
  float* ostage = reinterpret_cast<float*>(smem + kOffTile);  // [16][512]
  float* mst = ostage + kNR * kRank;
  float* lst = mst + kNR;
  if (warp < 4) {
    // this CTA's state over its tokens: O^T block c lanes = columns 128 c + 32 warp + lane
    const bool use_o = have && any_pv;
#pragma unroll
    for (int c = 0; c < kQuad; ++c) {
      float v[16];
      if (use_o) {
        tc_fence_after();
        tmem_ld16(tmem + tmem_lane_base(warp) + 2 * kNR + c * kNR, v);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) v[jj] = 0.f;
      }
      const int d = c * 128 + warp * 32 + lane;
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) ostage[jj * kRank + d] = v[jj];
    }
    if (warp == qr) {
#pragma unroll
      for (int r = 0; r < kNR; ++r) {
        float v = lsum[r];
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        if (lane == r) {
          mst[r] = use_o ? mr[r] : -INFINITY;
          lst[r] = use_o ? v : 0.f;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  // the cluster's result goes to the chunk's slot, or, when the chunk is spread over several
  // clusters, to this cluster's sub-partial slot of the workspace
  if (subs > 1)
    cluster_combine_to(p, w, ostage, mst, lst, tid, kThreads, p.ws_partials, p.ws_lse,
                       static_cast<long long>(blockIdx.y));
  else
    cluster_combine_to(p, w, ostage, mst, lst, tid, kThreads, p.partials, p.lse, static_cast<long long>(w.slot));
  if (subs > 1) merge_sub_partials(p, w, chunk, subs, &sm->last_cluster, tid, kThreads);
  cluster_sync();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

cudaError_t prepare(int cluster) {
  static bool smem_set = false, np_set = false;
  const void* fn = reinterpret_cast<const void*>(&mla_partial_quad_kernel);
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

bool quad_supports(int total_rows, bool bf16, int cluster) {
  return total_rows <= kNR && !bf16 && (cluster == 4 || cluster == 8 || cluster == 16);
}

cudaError_t launch_partial_quad(const CUtensorMap& tm_pages, const CUtensorMap& tm_kpe, const PartialParams& p,
                                int num_chunks, int cluster, cudaStream_t stream) {
  cudaError_t e = prepare(cluster);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster, num_chunks * (p.subs > 1 ? p.subs : 1), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_partial_quad_kernel, tm_pages, tm_kpe, p);
}

int quad_max_active_clusters(int cluster) {
  if (prepare(cluster) != cudaSuccess) {
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
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(&mla_partial_quad_kernel), &cfg) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t quad_read_clear_error(uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_device_error, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(uint32_t));
}

}  // namespace mla
