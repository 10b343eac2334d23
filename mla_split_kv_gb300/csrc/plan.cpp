// Partition planner (host only, no GPU access).
//
// "[kernel] Wire MLA split-KV decode" (vllm-metal PR #601), *What changed*:
// host dispatch takes the split path only in conservative cases -- long enough
// context, 2 to 8 partitions, bounded temporary memory -- and the review asks
// for these thresholds to live in a device-aware split-plan helper. "feat(core):
// matrix-absorbed MLA decode over a compressed-latent KV cache", *What
// changed*: `MlaSplitPlan` cuts the latent range into chunks.
//
// Here a partition is one thread-block cluster of C CTAs (the CTAs split the
// partition's tokens and combine on chip), so the plan is sized against the
// number of co-resident clusters of the partial kernel: partitions are shared
// out over requests in proportion to their lengths so that one wave of
// clusters covers all of them. With the paired 16-row kernel a partition may
// also span k clusters (combined through a workspace), so that the 2..8
// partitions of one request still fill the device.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "kernels.h"
#include "mla_split_kv.h"

namespace {

int64_t chunk_len(int64_t L, int64_t P, int64_t bs) {
  const int64_t per = (L + P - 1) / P;
  int64_t C = ((per + bs - 1) / bs) * bs;
  return C < bs ? bs : C;
}

// Largest P' <= P whose chunks are all non-empty under the chunk rule.
int64_t no_empty_chunks(int64_t L, int64_t P, int64_t bs) {
  while (P > 1 && (P - 1) * chunk_len(L, P, bs) >= L) --P;
  return P;
}

struct Candidate {
  int cluster = 1;
  int64_t subs = 1;     // clusters per partition
  std::vector<int64_t> parts;
  int64_t active = -1;  // CTAs busy in the first wave
  double cost_us = 0;   // modelled time (single request on the paired kernel)
};

constexpr int64_t kMaxSubs = 16;       // clusters per partition (the kernel's final merge reads at most 16)
constexpr int64_t kPairTileTokens = 128;
// Time model of the paired kernel for one request, fitted to steady-state layer-call times measured
// on GB300 (back-to-back calls over caches larger than L2) over partition counts, cluster sizes and
// spreads at 32K-128K tokens: a call takes about 1.75 us per 128-token tile of its busiest CTA
// pair (a chunk's tiles are split evenly over its k * C/2 pairs) plus a fixed part common to every
// plan. With the pairs' parts merged as entries (MLA_MERGE_ENTRIES) a spread costs nothing more,
// except 0.6 us per further round of 96 entries in the merge; when each chunk's parts are first
// merged into the chunk's partial by its last CTA (MLA_MERGE_PARTIALS), a spread adds a ticket +
// merge tail of ~6 us plus ~0.3 us per sub-partial for a 2-CTA cluster (the merge work per CTA
// scales with k / C).
constexpr double kTileUs = 1.75, kSpreadTailUs = 6.0, kMergeUsPerSub = 0.3;
constexpr double kEntriesRoundUs = 0.6;
constexpr int64_t kEntriesPerRound = 96;

double paired_cost_us(int64_t L, int64_t P, int64_t k, int C, int32_t merge_path, int64_t bs) {
  const int64_t pairs_per_chunk = k * (C / 2);
  const int64_t chunk_tiles = (chunk_len(L, P, bs) + kPairTileTokens - 1) / kPairTileTokens;
  const int64_t per_pair = (chunk_tiles + pairs_per_chunk - 1) / pairs_per_chunk;
  double t = static_cast<double>(per_pair) * kTileUs;
  if (merge_path == MLA_MERGE_ENTRIES) {
    const int64_t entries = P * pairs_per_chunk;
    t += kEntriesRoundUs * static_cast<double>((entries + kEntriesPerRound - 1) / kEntriesPerRound - 1);
  } else if (k > 1) {
    t += kSpreadTailUs + kMergeUsPerSub * static_cast<double>(k) * 2.0 / static_cast<double>(C);
  }
  return t;
}

}  // namespace

extern "C" mla_status_t mla_plan(const int32_t* context_lens_host, int32_t B, int32_t num_heads, int32_t q_len,
                                 int32_t block_size, const mla_device_info_t* dev, mla_plan_t* plan) {
  if (context_lens_host == nullptr || dev == nullptr || plan == nullptr) return MLA_ERR_INVALID_ARG;
  if (B < 1 || B > 65535) return MLA_ERR_INVALID_ARG;
  if (num_heads != 16 && num_heads != 64 && num_heads != 128) return MLA_ERR_UNSUPPORTED;
  if (q_len < 1 || q_len > MLA_MAX_Q_LEN) return MLA_ERR_UNSUPPORTED;
  if (block_size != 16 && block_size != 32 && block_size != 64) return MLA_ERR_UNSUPPORTED;
  if (plan->dtype != MLA_F16 && plan->dtype != MLA_BF16 && plan->dtype != MLA_E4M3) return MLA_ERR_UNSUPPORTED;
  if (plan->capacity < 0 || plan->max_partitions < 0 || plan->min_partitions < 0 || plan->split_min_tokens < 0)
    return MLA_ERR_INVALID_ARG;
  if (plan->merge_path != MLA_MERGE_ENTRIES && plan->merge_path != MLA_MERGE_PARTIALS) return MLA_ERR_INVALID_ARG;
  const int32_t merge_path = plan->merge_path;
  if (dev->num_sms < 1) return MLA_ERR_INVALID_ARG;
  for (int32_t b = 0; b < B; ++b)
    if (context_lens_host[b] < 0) return MLA_ERR_INVALID_ARG;

  const int64_t maxP = plan->max_partitions ? plan->max_partitions : 8;
  const int64_t minP = std::min<int64_t>(plan->min_partitions ? plan->min_partitions : 2, maxP);
  const int64_t split_min = plan->split_min_tokens ? plan->split_min_tokens : 4096;
  if (maxP < 1 || maxP > 1024) return MLA_ERR_INVALID_ARG;

  const int rows = num_heads * q_len;
  // more than 16 rows: one CTA pair (a cluster of 2) per 128 rows, the last group padded
  const bool many_rows = mla::mh_supports(rows, 2);
  const int nr = many_rows ? 128 : mla::tc_rows_per_cta(rows, plan->dtype == MLA_BF16);
  const int64_t row_groups = (rows + nr - 1) / nr;

  int64_t split_tokens = 0, n_split = 0;
  for (int32_t b = 0; b < B; ++b)
    if (context_lens_host[b] >= split_min) {
      split_tokens += context_lens_host[b];
      ++n_split;
    }

  Candidate best;
  // 16 rows run on the paired kernel whenever the device has CTA pairs: a
  // partition's tiles stream through three slots on two SMs, several times the 64-token kernel's
  // rate, so clusters of one are not candidates then (for a batch they would tie on busy CTAs)
  const bool paired_ok = mla::tc128_supports(rows, plan->dtype == MLA_BF16, 2) && dev->max_clusters[1] > 0;
  // one long request on the paired kernel: candidates compared by the time model
  const bool paired_single = (B == 1 && n_split == 1 && paired_ok);
  for (int k = 0; k < 5; ++k) {
    const int C = 1 << k;
    const int64_t slots = dev->max_clusters[k];
    if (slots <= 0) continue;
    if (paired_ok && C == 1) continue;  // the paired kernel needs a pair of CTAs
    if (plan->dtype == MLA_E4M3 && C == 1) continue;  // so do E4M3 caches, always
    if (many_rows && C != 2) continue;      // the 128-row kernel runs on CTA pairs
    Candidate cand;
    cand.cluster = C;
    cand.parts.assign(B, 1);
    const int64_t budget = std::max<int64_t>(B, slots / row_groups);
    const int64_t spare = budget - (B - n_split);  // partitions left for the split requests
    bool ok = true;
    if (n_split > 0) {
      // proportional share, floor, then largest remainder, all clamped
      std::vector<std::pair<double, int32_t>> rem;
      int64_t used = 0;
      for (int32_t b = 0; b < B; ++b) {
        const int64_t L = context_lens_host[b];
        if (L < split_min) continue;
        const double share = static_cast<double>(spare) * static_cast<double>(L) / static_cast<double>(split_tokens);
        int64_t P = static_cast<int64_t>(share);
        P = std::max(minP, std::min(maxP, std::max<int64_t>(P, 1)));
        cand.parts[b] = P;
        used += P;
        rem.push_back({share - static_cast<double>(static_cast<int64_t>(share)), b});
      }
      std::stable_sort(rem.begin(), rem.end(), [](const auto& a, const auto& c) { return a.first > c.first; });
      for (size_t j = 0; j < rem.size() && used < spare; ++j) {
        const int32_t b = rem[j].second;
        if (cand.parts[b] < maxP) {
          ++cand.parts[b];
          ++used;
        }
      }
      for (int32_t b = 0; b < B; ++b) {
        const int64_t L = context_lens_host[b];
        if (L < split_min) continue;
        cand.parts[b] = no_empty_chunks(L, cand.parts[b], block_size);
        // every CTA of the cluster should get at least one 64-token tile
        if (C > 1 && chunk_len(L, cand.parts[b], block_size) < static_cast<int64_t>(C) * mla::kTileTokens) ok = false;
      }
    }
    if (!ok) continue;
    int64_t N = 0;
    for (int32_t b = 0; b < B; ++b) N += cand.parts[b];
    // spread each partition over k clusters when the paired kernel runs and a wave has room,
    // every CTA pair keeping at least one 128-token tile of its partition
    auto largest_k = [&](const std::vector<int64_t>& parts, int64_t n) -> int64_t {
      int64_t k = std::min<int64_t>(kMaxSubs, slots / (n * row_groups));
      for (; k > 1; --k) {
        bool fits = true;
        for (int32_t b = 0; b < B && fits; ++b) {
          const int64_t L = context_lens_host[b];
          const int64_t len = (parts[b] > 1) ? chunk_len(L, parts[b], block_size) : L;
          if (len < k * (C / 2) * kPairTileTokens) fits = false;
        }
        if (fits) break;
      }
      return std::max<int64_t>(1, k);
    };
    if (mla::tc128_supports(rows, plan->dtype == MLA_BF16, C) && N * row_groups < slots) {
      cand.subs = largest_k(cand.parts, N);
      if (paired_single) {
        // one long request: among the allowed partition counts and spreads take the fastest by the
        // time model (ties: more CTA pairs busy, then fewer clusters per partition)
        const int64_t L = context_lens_host[0];
        double best_cost = paired_cost_us(L, N, cand.subs, C, merge_path, block_size);
        std::vector<int64_t> parts1(1);
        for (int64_t P1 = minP; P1 <= maxP; ++P1) {
          parts1[0] = no_empty_chunks(L, P1, block_size);
          if (parts1[0] != P1 || P1 * row_groups > slots) continue;
          for (int64_t k1 = largest_k(parts1, P1); k1 >= 1; --k1) {
            const double c1 = paired_cost_us(L, P1, k1, C, merge_path, block_size);
            const int64_t pairs1 = P1 * k1, pairs0 = cand.parts[0] * cand.subs;
            const bool tie = c1 < best_cost + 1e-9 && c1 > best_cost - 1e-9;
            if (c1 < best_cost - 1e-9 || (tie && (pairs1 > pairs0 || (pairs1 == pairs0 && k1 < cand.subs)))) {
              best_cost = c1;
              cand.parts[0] = P1;
              cand.subs = k1;
            }
          }
        }
        N = cand.parts[0];
      }
    }
    // the time model assumes one wave: a launch whose clusters cannot all be co-resident (the
    // partition floor exceeding the device's clusters of this size) is not a candidate
    if (paired_single && N * cand.subs * row_groups > slots) continue;
    if (paired_single) cand.cost_us = paired_cost_us(context_lens_host[0], N, cand.subs, C, merge_path, block_size);
    cand.active = std::min<int64_t>(N * row_groups * cand.subs, slots) * C;
    if (paired_single) {
      // the modelled fastest; on a tie the smaller cluster (visited first)
      if (best.active < 0 || cand.cost_us < best.cost_us - 1e-9) best = cand;
    } else if (cand.active > best.active || (cand.active == best.active && cand.subs < best.subs)) {
      // more busy CTAs wins; on a tie, fewer clusters per partition, then the smaller cluster
      best = cand;
    }
  }
  if (best.active < 0) {  // no cluster size usable: one CTA per partition, no split
    best = Candidate();
    best.cluster = 1;
    best.parts.assign(B, 1);
  }

  int64_t N = 0;
  for (int32_t b = 0; b < B; ++b) N += best.parts[b];
  if (N > 65535) return MLA_ERR_UNSUPPORTED;
  plan->num_chunks = static_cast<int32_t>(N);
  plan->cluster_ctas = best.cluster;
  plan->kernel = MLA_KERNEL_TC;
  plan->clusters_per_chunk = static_cast<int32_t>(best.subs);
  if (N > plan->capacity) return MLA_ERR_CAPACITY;
  if (plan->chunks == nullptr || plan->o_indptr == nullptr) return MLA_ERR_INVALID_ARG;

  int32_t n = 0;
  for (int32_t b = 0; b < B; ++b) {
    plan->o_indptr[b] = n;
    const int64_t L = context_lens_host[b];
    const int64_t P = best.parts[b];
    const int64_t Cl = chunk_len(L, P, block_size);
    for (int64_t p = 0; p < P; ++p) {
      const int64_t t0 = std::min(p * Cl, L), t1 = std::min((p + 1) * Cl, L);
      plan->chunks[n] = mla_chunk_t{b, static_cast<int32_t>(t0), static_cast<int32_t>(t1), n};
      ++n;
    }
  }
  plan->o_indptr[B] = n;
  return MLA_OK;
}
