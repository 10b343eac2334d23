// Tensor-core partial-decode kernel for CTAs of 16 query rows (fp16), sm_103a.
//
// The operation is the one of the other partial kernels ("feat(core):
// matrix-absorbed MLA decode over a compressed-latent KV cache", *What
// changed*: SDPA(q_absorbed, ckv, ckv, scale, mask = scale * q_pe @ kpe^T),
// each chunk yielding a normalized partial and its log2 LSE).
//
// 16 query rows (the heads of a one-token decode) are too few for the tensor
// core's M side, so both products put tokens / latent columns on M=128 and the
// 16 rows on N:
//   S^T[tok, row] = [ckv | kpe][tok, 0:576] . Q^T      M=128 tokens, N=16, K=576
//   O^T[d, row]  += ckv^T[d, tok] . P^T[tok, row]      M=128 (x4), N=16, K=128
// At N=16 every tcgen05.mma costs about the same fixed time, so a tile of 128
// tokens (68 MMAs) is used rather than 64 (52 MMAs for half the tokens). A
// 128-token tile is 144 KB, more than half of shared memory, so the latent is
// staged in a ring of five 32 KB "pair slots" (a pair = two 64-column ckv boxes
// = one 128-column block of the latent for 128 tokens) plus two 16 KB kpe
// slots. A pair slot is released as soon as the PV block that reads it is
// done, and the MMA warp issues, per tile i: the head of the score product of
// tile i (kpe and pair 0), the PV product of tile i-1, then the tail of the
// score product of tile i (pairs 1..3). Reloads of released slots then overlap
// MMA work, and the softmax of tile i-1 overlaps the head of tile i.
//
// TMA issue costs about the same per instruction whatever the box size, so the
// loads are spread over eleven producer warps: warps 5+2s and 6+2s own the two
// 64-column boxes of pair slot s (every use of a slot is issued by the same two
// warps, in order) and warp 15 loads kpe. Each producer also prefetches its
// boxes of the tile after next into L2.
//
// Warp roles (512 threads): warps 0-3 softmax / O rescale / epilogue, warp 4
// TMEM owner + MMA issuer, warps 5-14 pair-slot producers, warp 15 kpe producer.
#include "device_common.cuh"

namespace mla {

namespace {

constexpr int kT = 128;                    // tokens per tile
constexpr int kNR = 16;                    // query rows per CTA
constexpr int kSlots = 5;                  // pair slots
constexpr int kBox128 = kT * 128;          // one 64-column box of 128 rows: 16 KB
constexpr int kPairBytes = 2 * kBox128;    // 32 KB
constexpr int kThreads = 16 * 32;
constexpr float kRescaleTau = 8.0f;

constexpr uint32_t kOffPair = 0;
constexpr uint32_t kOffKpe = kSlots * kPairBytes;               // 160 KB
constexpr uint32_t kOffQ = kOffKpe + 2 * kBox128;               // 192 KB
constexpr uint32_t kQChunk = kNR * 128;                         // 2 KB
constexpr uint32_t kOffP = kOffQ + 9 * kQChunk;                 // 210 KB
constexpr uint32_t kPBuf = 2 * kNR * 128;                       // P^T [16 x 128 tokens]: two 64-token atoms
constexpr uint32_t kOffSmall = kOffP + 2 * kPBuf;               // 218 KB
constexpr uint32_t kSmem = kOffSmall + 2048 + 1024;             // + alignment slack
constexpr uint32_t kTmemCols = 128;                             // S^T 2x16 + O^T 4x16
static_assert(kSmem <= 232448, "shared memory per CTA");

struct Small {
  uint64_t pfull[kSlots], pempty[kSlots], kfull[2], kempty[2], sfull[2], sfree[2], ppfull[2], pvdone[2], drain;
  uint32_t tmem_base;
  int32_t abort_flag;
  float red[4][kNR];
  float mref[kNR];
  float alpha[kNR];
};
static_assert(sizeof(Small) <= 2048, "small smem region");

__device__ __forceinline__ uint32_t tmem_lane_base(int warp) { return static_cast<uint32_t>(32 * (warp & 3)) << 16; }
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

// Pair j of tile i lives in slot (4i + j) % 5; it is that slot's use number (4i + j) / 5.
__device__ __forceinline__ int slot_of(int i, int j) { return (4 * i + j) % kSlots; }
__device__ __forceinline__ int use_of(int i, int j) { return (4 * i + j) / kSlots; }

__global__ void __launch_bounds__(kThreads, 1)
    mla_partial_tc128_kernel(const __grid_constant__ CUtensorMap tm_ckv, const __grid_constant__ CUtensorMap tm_kpe,
                             const PartialParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* qs = smem + kOffQ;
  uint8_t* ps = smem + kOffP;
  Small* sm = reinterpret_cast<Small*>(smem + kOffSmall);
  volatile int32_t* abort_flag = &sm->abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const CtaWork w = cta_work(p, kNR, kT);
  const int ntiles = (w.sub1 - w.sub0 + kT - 1) / kT;
  const int rows_total = p.q_len * p.H;

  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&sm->pfull[s], 2);  // one arrival per box-half producer
      mbar_init(&sm->pempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm->kfull[b], 1);
      mbar_init(&sm->kempty[b], 1);
      mbar_init(&sm->sfull[b], 1);
      mbar_init(&sm->sfree[b], 4);
      mbar_init(&sm->ppfull[b], 4);
      mbar_init(&sm->pvdone[b], 1);
    }
    mbar_init(&sm->drain, 1);
    sm->abort_flag = 0;
    fence_mbar_init();
  }
  if (tid < kNR) sm->mref[tid] = -INFINITY;
  if (warp == 4) {
    tmem_alloc(&sm->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp < 4) {  // Q^T: 16 rows x 576, K-major, 9 swizzled [16 x 64] chunks
    for (int idx = tid; idx < kNR * (kQkDim / 8); idx += 128) {
      const int r = idx / (kQkDim / 8), k = (idx % (kQkDim / 8)) * 8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (r < w.nrows) {
        const long long row = static_cast<long long>(w.b) * rows_total + w.row0 + r;
        v = (k < kRank) ? *reinterpret_cast<const uint4*>(p.q_abs + row * kRank + k)
                        : *reinterpret_cast<const uint4*>(p.q_pe + row * kRope + (k - kRank));
      }
      *reinterpret_cast<uint4*>(qs + (k / kBoxCols) * kQChunk + sw128_offset(r, k % kBoxCols)) = v;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;

  if (warp >= 5) {
    // ------------------------------------------------------------------ producers
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
    const bool kpe_warp = (warp == 15);
    const int s = (warp - 5) >> 1;  // pair slot owned by this warp
    const int half = (warp - 5) & 1;  // which 64-column box of the pair
    int issued_q = -1;       // last (tile, pair) index this warp loaded
    for (int i = 0; i < ntiles; ++i) {
      int pg0, npg;
      tile_pages(i, &pg0, &npg);
      int j = -1;
      if (kpe_warp) {
        j = 8;  // kpe box
      } else {
        const int jj = ((s - 4 * i) % kSlots + kSlots) % kSlots;
        if (jj < 4) j = jj;
      }
      if (j < 0) continue;  // this slot is not used by tile i
      // wait until the previous use of the destination is released
      int ok = 1;
      if (lane == 0) {
        if (kpe_warp) {
          if (i >= 2) ok = mbar_wait(&sm->kempty[i & 1], ((i >> 1) - 1) & 1, p.timeout_ns);
        } else {
          const int u = use_of(i, j);
          if (u >= 1) ok = mbar_wait(&sm->pempty[s], (u - 1) & 1, p.timeout_ns);
        }
        ok = ok && !*abort_flag;
        if (!ok) *abort_flag = 1;
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      int pids[kT / 16];
#pragma unroll
      for (int k = 0; k < kT / 16; ++k) pids[k] = (k < npg) ? page_of(pg0 + k) : -1;
      if (lane == 0) {
        if (kpe_warp) {
          uint8_t* dst = smem + kOffKpe + (i & 1) * kBox128;
          mbar_arrive_expect_tx(&sm->kfull[i & 1], static_cast<uint32_t>(npg * p.bs * 128));
          for (int k = 0; k < npg; ++k) tma_load_2d(dst + k * p.bs * 128, &tm_kpe, 0, pids[k] * p.bs, &sm->kfull[i & 1], pol);
        } else {
          uint8_t* dst = smem + kOffPair + s * kPairBytes + half * kBox128;
          mbar_arrive_expect_tx(&sm->pfull[s], static_cast<uint32_t>(npg * p.bs * 128));
          for (int k = 0; k < npg; ++k)
            tma_load_2d(dst + k * p.bs * 128, &tm_ckv, (2 * j + half) * kBoxCols, pids[k] * p.bs, &sm->pfull[s], pol);
        }
      }
      issued_q = i;
      // the same boxes of the tile after next, into L2
      if (i + 2 < ntiles) {
        int qg0, qn;
        tile_pages(i + 2, &qg0, &qn);
        for (int k = 0; k < qn; ++k) {
          const int pid = page_of(qg0 + k);
          if (lane == 0 && pid >= 0) {
            if (kpe_warp) {
              tma_prefetch_l2_2d(&tm_kpe, 0, pid * p.bs);
            } else {
              tma_prefetch_l2_2d(&tm_ckv, (2 * j + half) * kBoxCols, pid * p.bs);
            }
          }
        }
      }
    }
    // after an abort, let this warp's last load land before shared memory is released
    if (lane == 0 && *abort_flag && issued_q >= 0) {
      if (kpe_warp) {
        mbar_wait(&sm->kfull[issued_q & 1], (issued_q >> 1) & 1, kDrainTimeoutNs);
      } else {
        const int jj = ((s - 4 * issued_q) % kSlots + kSlots) % kSlots;
        mbar_wait(&sm->pfull[s], use_of(issued_q, jj) & 1, kDrainTimeoutNs);
      }
    }
  } else if (warp == 4) {
    // ------------------------------------------------------------------ MMA issuer
    const uint32_t idesc_s = idesc_f16_f32(128, kNR, false, false, false);
    const uint32_t idesc_o = idesc_f16_f32(128, kNR, false, true, false);
    const uint64_t q_desc = smem_desc_sw128(smem_u32(qs), 16, 1024);
    const uint64_t p_desc = smem_desc_sw128(smem_u32(ps), 16, 1024);
    const uint32_t pair_base = smem_u32(smem + kOffPair), kpe_base = smem_u32(smem + kOffKpe);
    bool alive = true;
    auto wait_lane0 = [&](uint64_t* bar, uint32_t parity) -> bool {
      int ok = 1;
      if (lane == 0) {
        ok = mbar_wait(bar, parity, p.timeout_ns) && !*abort_flag;
        if (!ok) *abort_flag = 1;
      }
      return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    // rows >= nvalid of a 128-row box: zero them so the A operand stays finite
    auto zero_tail = [&](uint8_t* box, int nvalid) {
      for (int x = lane; x < (kT - nvalid) * 8; x += 32)
        *reinterpret_cast<uint4*>(box + nvalid * 128 + x * 16) = make_uint4(0u, 0u, 0u, 0u);
    };
    // score MMAs over box c (c < 8: ckv column block c, c = 8: kpe) of tile i
    auto score_box = [&](int i, int c, bool first) {
      const uint32_t a = (c < 8) ? pair_base + slot_of(i, c >> 1) * kPairBytes + (c & 1) * kBox128
                                 : kpe_base + (i & 1) * kBox128;
      const uint64_t ad = smem_desc_sw128(a, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        umma_f16_ss(tmem + (i & 1) * kNR, desc_add(ad, kk * 32), desc_add(q_desc, c * kQChunk + kk * 32), idesc_s,
                    (first && kk == 0) ? 0u : 1u);
    };
    auto pair_ready = [&](int i, int j, int nvalid) -> bool {
      if (!wait_lane0(&sm->pfull[slot_of(i, j)], use_of(i, j) & 1)) return false;
      if (nvalid < kT) {
        uint8_t* pr = smem + kOffPair + slot_of(i, j) * kPairBytes;
        zero_tail(pr, nvalid);
        zero_tail(pr + kBox128, nvalid);
        fence_proxy_async_smem();
        __syncwarp();
      }
      return true;
    };
    for (int i = 0; i <= ntiles && alive; ++i) {
      const int nvalid = (i < ntiles) ? min(kT, w.sub1 - (w.sub0 + i * kT)) : 0;
      if (i < ntiles) {  // head of the score product: kpe, pair 0
        if (!wait_lane0(&sm->kfull[i & 1], (i >> 1) & 1)) break;
        if (nvalid < kT) {
          zero_tail(smem + kOffKpe + (i & 1) * kBox128, nvalid);
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (i >= 2 && !wait_lane0(&sm->sfree[i & 1], ((i >> 1) - 1) & 1)) break;
        if (!pair_ready(i, 0, nvalid)) break;
        if (lane == 0) {
          tc_fence_after();
          score_box(i, 8, true);
          score_box(i, 0, false);
          score_box(i, 1, false);
        }
        __syncwarp();
      }
      if (i >= 1) {  // PV of the previous tile, releasing its pair slots block by block
        const int j = i - 1;
        if (!wait_lane0(&sm->ppfull[j & 1], (j >> 1) & 1)) break;
        if (lane == 0) {
          tc_fence_after();
          const uint64_t pb = desc_add(p_desc, (j & 1) * kPBuf);
#pragma unroll
          for (int blk = 0; blk < 4; ++blk) {
            const uint64_t a0 = smem_desc_sw128(pair_base + slot_of(j, blk) * kPairBytes, kBox128, 1024);
#pragma unroll
            for (int ks = 0; ks < kT / 16; ++ks)
              umma_f16_ss(tmem + 2 * kNR + blk * kNR, desc_add(a0, ks * 16 * 128),
                          desc_add(pb, (ks >> 2) * (kNR * 128) + (ks & 3) * 32), idesc_o, (j > 0 || ks > 0) ? 1u : 0u);
            umma_commit(&sm->pempty[slot_of(j, blk)]);
          }
          umma_commit(&sm->pvdone[j & 1]);
        }
        __syncwarp();
      }
      if (i < ntiles) {  // tail of the score product: pairs 1..3
        bool ok = true;
        for (int jp = 1; jp < 4 && ok; ++jp) {
          ok = pair_ready(i, jp, nvalid);
          if (ok && lane == 0) {
            tc_fence_after();
            score_box(i, 2 * jp, false);
            score_box(i, 2 * jp + 1, false);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) {
          umma_commit(&sm->sfull[i & 1]);
          umma_commit(&sm->kempty[i & 1]);
        }
        __syncwarp();
      }
    }
    if (lane == 0) {  // every MMA issued so far has completed before TMEM is read or freed
      umma_commit(&sm->drain);
      mbar_wait(&sm->drain, 0, kDrainTimeoutNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax (warps 0-3)
    // Thread (warp, lane) owns token 32*warp + lane of each tile (M=128 layout of S^T).
    float lsum[kNR];
#pragma unroll
    for (int r = 0; r < kNR; ++r) lsum[r] = 0.f;
    const int tl = 32 * warp + lane;
    const int causal_floor = p.causal ? w.L - p.q_len + w.row0 / p.H : 0x7fffffff;
    for (int i = 0; i < ntiles; ++i) {
      const int buf = i & 1;
      const int tok0 = w.sub0 + i * kT;
      const int nvalid = min(kT, w.sub1 - tok0);
      const bool masked_tile = (nvalid < kT) || (tok0 + kT - 1 > causal_floor) || (w.nrows < kNR);
      float x[kNR];
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&sm->sfull[buf], (i >> 1) & 1, p.timeout_ns);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      bool need_local = false;
      if (ok) {
        tc_fence_after();
        tmem_ld16(tmem + tmem_lane_base(warp) + buf * kNR, x);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->sfree[buf]);
        const int t = tok0 + tl;
#pragma unroll
        for (int r = 0; r < kNR; ++r) {
          bool vis = true;
          if (masked_tile) {
            vis = (tl < nvalid) && (r < w.nrows);
            if (p.causal) vis = vis && (t <= w.L - p.q_len + (w.row0 + r) / p.H);
          }
          x[r] = vis ? x[r] * p.scale_log2 : -INFINITY;
          need_local |= x[r] > sm->mref[r] + kRescaleTau;
        }
      } else {
#pragma unroll
        for (int r = 0; r < kNR; ++r) x[r] = -INFINITY;
        if (lane == 0) *abort_flag = 1;
      }
      if (named_bar_sync_or(1, 128, need_local || *abort_flag != 0)) {
        if (named_bar_sync_or(1, 128, *abort_flag != 0)) break;
        // rare path: move the reference max, rescale O^T and the row sums
#pragma unroll
        for (int r = 0; r < kNR; ++r) {
          float v = x[r];
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
          if (lane == 0) sm->red[warp][r] = v;
        }
        named_bar_sync(1, 128);
        if (tid < kNR) {
          const float mprev = sm->mref[tid];
          const float tmax = fmaxf(fmaxf(sm->red[0][tid], sm->red[1][tid]), fmaxf(sm->red[2][tid], sm->red[3][tid]));
          const float mnew = fmaxf(mprev, tmax);
          sm->alpha[tid] = (mnew == -INFINITY) ? 1.f : exp2f(mprev - mnew);
          sm->mref[tid] = mnew;
        }
        named_bar_sync(1, 128);
        if (i >= 1) {  // PV(i-1) must be complete before O^T is rescaled
          int ok2 = 1;
          if (lane == 0) ok2 = mbar_wait(&sm->pvdone[(i - 1) & 1], ((i - 1) >> 1) & 1, p.timeout_ns);
          if (__shfl_sync(0xffffffffu, ok2, 0)) {
            tc_fence_after();
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
              float v[16];
              const uint32_t a = tmem + tmem_lane_base(warp) + 2 * kNR + blk * kNR;
              tmem_ld16(a, v);
              tmem_wait_ld();
#pragma unroll
              for (int jj = 0; jj < 16; ++jj) v[jj] *= sm->alpha[jj];
              tmem_st16(a, v);
            }
            tmem_wait_st();
          } else if (lane == 0) {
            *abort_flag = 1;
          }
        }
#pragma unroll
        for (int r = 0; r < kNR; ++r) lsum[r] *= sm->alpha[r];
      }
      if (i >= 2) {  // P^T buffer `buf` was last read by PV(i-2)
        int ok3 = 1;
        if (lane == 0) ok3 = mbar_wait(&sm->pvdone[buf], ((i >> 1) - 1) & 1, p.timeout_ns);
        if (!__shfl_sync(0xffffffffu, ok3, 0) && lane == 0) *abort_flag = 1;
      }
      {  // probabilities -> P^T (fp16, K-major, two swizzled 64-token atoms) and row sums
        uint8_t* pb = ps + buf * kPBuf + (tl >> 6) * (kNR * 128);
#pragma unroll
        for (int r = 0; r < kNR; ++r) {
          const float pr = (x[r] == -INFINITY) ? 0.f : exp2f(x[r] - sm->mref[r]);
          const uint16_t hv = f2h<false>(pr);
          lsum[r] += h2f<false>(hv);
          *reinterpret_cast<uint16_t*>(pb + sw128_offset(r, tl & 63)) = hv;
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->ppfull[buf]);
    }
    const bool aborted = named_bar_sync_or(1, 128, *abort_flag != 0);
    if (ntiles > 0 && !aborted) {
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&sm->pvdone[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, p.timeout_ns);
      if (!__shfl_sync(0xffffffffu, ok, 0) && lane == 0) *abort_flag = 1;
    }
#pragma unroll
    for (int r = 0; r < kNR; ++r) {
      float v = lsum[r];
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      if (lane == 0) sm->red[warp][r] = v;
    }
    named_bar_sync(1, 128);
  }
  __syncthreads();  // all roles done: the pair slots are free for staging
  const bool have = (ntiles > 0) && !*abort_flag;
  float* ostage = reinterpret_cast<float*>(smem + kOffPair);  // [16][512]
  float* mst = ostage + kNR * kRank;
  float* lst = mst + kNR;
  if (warp < 4) {
    if (have) {
      tc_fence_after();
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        float v[16];
        tmem_ld16(tmem + tmem_lane_base(warp) + 2 * kNR + blk * kNR, v);
        tmem_wait_ld();
        const int d = blk * 128 + warp * 32 + lane;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) ostage[jj * kRank + d] = v[jj];
      }
    } else {
      for (int idx = tid; idx < kNR * kRank; idx += 128) ostage[idx] = 0.f;
    }
    if (tid < kNR) {
      mst[tid] = have ? sm->mref[tid] : -INFINITY;
      lst[tid] = have ? (sm->red[0][tid] + sm->red[1][tid]) + (sm->red[2][tid] + sm->red[3][tid]) : 0.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  cluster_combine(p, w, ostage, mst, lst, tid, kThreads);
  cluster_sync();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

cudaError_t prepare(int cluster) {
  static bool smem_set = false, np_set = false;
  const void* fn = reinterpret_cast<const void*>(&mla_partial_tc128_kernel);
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

bool tc128_supports(int total_rows, bool bf16) { return total_rows <= kNR && !bf16; }

cudaError_t launch_partial_tc128(const CUtensorMap& tm_ckv, const CUtensorMap& tm_kpe, const PartialParams& p,
                                 int num_chunks, int cluster, cudaStream_t stream) {
  cudaError_t e = prepare(cluster);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster, num_chunks, 1);
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
  return cudaLaunchKernelEx(&cfg, mla_partial_tc128_kernel, tm_ckv, tm_kpe, p);
}

int tc128_max_active_clusters(int cluster) {
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
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(&mla_partial_tc128_kernel), &cfg) !=
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
