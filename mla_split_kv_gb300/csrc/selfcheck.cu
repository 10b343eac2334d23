// mla_selfcheck: one decode through the public calls on a built-in case whose
// result is known in closed form, so that a user can check a device and a
// build without any reference implementation.
//
// The case: two requests (6000 and 700 tokens, the last page of each partial),
// 16 heads, pages of 32 tokens scattered over the pool by a fixed permutation,
// pool pages that no request owns filled with 1000.0. The latent of token t is
// f(t, d) = ((13 t + 7 d) mod 64 - 32) / 8, exact in fp16 and bf16.
//  - heads 0..7 ("rope needles"): q_pe[h] is one-hot on column j_h and
//    kpe[t_h, j_h] = 16, every other kpe entry 0;
//  - heads 8..14 ("latent needles"): q_absorbed[h] is one-hot on column c_h and
//    ckv[t_h, c_h] = 16 (every other latent entry is at most 4 in magnitude);
//  - head 15: q_absorbed = q_pe = 0, every score is 0.
// With scale 4 a needle scores 64 against at most 16 elsewhere, so every other
// weight is below 2^-69 relative and vanishes in fp32: the output row of a
// needle head is the needle token's latent row, exactly, with base-2 LSE
// 64 log2(e); head 15 is the plain mean of the request's latent rows with LSE
// log2(L) (softmax of equal scores). One needle of each request sits on its
// last token. The columns j_h, c_h fall in both 256-column halves of the latent
// and both 32-column halves of the rope key. The check runs the planner's
// plan with the default kernel choice and again on the CUDA-core kernel, in
// fp16 and bf16.
#include <cmath>
#include <cstring>
#include <vector>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "mla_split_kv.h"

namespace {

constexpr int kB = 2, kH = 16, kBs = 32, kRank = MLA_KV_LORA_RANK, kRope = MLA_ROPE_DIM;
constexpr int kLens[kB] = {6000, 700};
constexpr int kPool = 256;  // pages in the pool; requests own ceil(L/32) = 188 + 22 of them
constexpr float kScale = 4.f, kNeedle = 16.f, kUnused = 1000.f;

int page_of(int logical) { return (logical * 37 + 11) % kPool; }  // 37 is odd: a permutation of 0..255
int rope_col(int h) { return 5 + 8 * h; }                          // heads 0..7: 5, 13, ..., 61
int latent_col(int h) { return 37 + 61 * (h - 8); }                // heads 8..14: 37 .. 403
int needle_token(int b, int h) {
  if (h == 14) return kLens[b] - 1;
  return b == 0 ? h * 397 + 123 : h * 43 + 5;
}
float latent(int t, int d) { return static_cast<float>((13 * t + 7 * d) % 64 - 32) * 0.125f; }

uint16_t to_bits(float x, int dtype) {
  uint16_t u;
  if (dtype == MLA_F16) {
    const __half h = __float2half_rn(x);
    std::memcpy(&u, &h, 2);
  } else {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    std::memcpy(&u, &h, 2);
  }
  return u;
}

// Device buffers of one check, freed on every return path.
struct Buffers {
  std::vector<void*> ptrs;
  ~Buffers() {
    for (void* p : ptrs) cudaFree(p);
  }
  template <class T>
  T* alloc(size_t bytes) {
    void* p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) return nullptr;
    ptrs.push_back(p);
    return static_cast<T*>(p);
  }
};

template <class T>
bool upload(T* dst, const std::vector<T>& src) {
  return cudaMemcpy(dst, src.data(), src.size() * sizeof(T), cudaMemcpyHostToDevice) == cudaSuccess;
}

mla_status_t run_one(int dtype, bool simt, float* max_err) {
  const int max_blocks = (kLens[0] + kBs - 1) / kBs;
  // host contents (floats) and the logical -> pool page map
  std::vector<float> ckv(static_cast<size_t>(kPool) * kBs * kRank, kUnused);
  std::vector<float> kpe(static_cast<size_t>(kPool) * kBs * kRope, 0.f);
  std::vector<int32_t> table(static_cast<size_t>(kB) * max_blocks, -1);  // past the last page: never read
  int next = 0;
  for (int b = 0; b < kB; ++b) {
    const int pages = (kLens[b] + kBs - 1) / kBs;
    for (int i = 0; i < pages; ++i) table[static_cast<size_t>(b) * max_blocks + i] = page_of(next++);
  }
  auto row = [&](int b, int t) {
    return static_cast<size_t>(table[static_cast<size_t>(b) * max_blocks + t / kBs]) * kBs + t % kBs;
  };
  for (int b = 0; b < kB; ++b)
    for (int t = 0; t < kLens[b]; ++t)
      for (int d = 0; d < kRank; ++d) ckv[row(b, t) * kRank + d] = latent(t, d);
  std::vector<float> q_abs(static_cast<size_t>(kB) * kH * kRank, 0.f), q_pe(static_cast<size_t>(kB) * kH * kRope, 0.f);
  for (int b = 0; b < kB; ++b) {
    for (int h = 0; h < 8; ++h) {
      q_pe[(static_cast<size_t>(b) * kH + h) * kRope + rope_col(h)] = 1.f;
      kpe[row(b, needle_token(b, h)) * kRope + rope_col(h)] = kNeedle;
    }
    for (int h = 8; h < 15; ++h) {
      q_abs[(static_cast<size_t>(b) * kH + h) * kRank + latent_col(h)] = 1.f;
      ckv[row(b, needle_token(b, h)) * kRank + latent_col(h)] = kNeedle;
    }
  }
  // expected rows and base-2 LSEs
  std::vector<double> want(static_cast<size_t>(kB) * kH * kRank), want_lse(static_cast<size_t>(kB) * kH);
  for (int b = 0; b < kB; ++b) {
    for (int h = 0; h < kH; ++h) {
      double* w = &want[(static_cast<size_t>(b) * kH + h) * kRank];
      if (h < 15) {
        const size_t r = row(b, needle_token(b, h));
        for (int d = 0; d < kRank; ++d) w[d] = ckv[r * kRank + d];
        want_lse[b * kH + h] = kScale * kNeedle / std::log(2.0);
      } else {
        for (int d = 0; d < kRank; ++d) w[d] = 0.0;
        for (int t = 0; t < kLens[b]; ++t)
          for (int d = 0; d < kRank; ++d) w[d] += ckv[row(b, t) * kRank + d];
        for (int d = 0; d < kRank; ++d) w[d] /= kLens[b];
        want_lse[b * kH + h] = std::log2(static_cast<double>(kLens[b]));
      }
    }
  }
  auto bits = [dtype](const std::vector<float>& v) {
    std::vector<uint16_t> out(v.size());
    for (size_t i = 0; i < v.size(); ++i) out[i] = to_bits(v[i], dtype);
    return out;
  };

  // plan
  mla_device_info_t dev;
  mla_status_t st = mla_device_query(-1, &dev);
  if (st != MLA_OK) return st;
  std::vector<mla_chunk_t> chunks(64);
  std::vector<int32_t> indptr(kB + 1);
  mla_plan_t plan;
  std::memset(&plan, 0, sizeof(plan));
  plan.dtype = dtype;
  plan.capacity = static_cast<int32_t>(chunks.size());
  plan.chunks = chunks.data();
  plan.o_indptr = indptr.data();
  st = mla_plan(kLens, kB, kH, 1, kBs, &dev, &plan);
  if (st != MLA_OK) return st;
  const int N = plan.num_chunks;
  chunks.resize(N);

  // device buffers
  Buffers buf;
  uint16_t* d_ckv = buf.alloc<uint16_t>(ckv.size() * 2);
  uint16_t* d_kpe = buf.alloc<uint16_t>(kpe.size() * 2);
  uint16_t* d_qa = buf.alloc<uint16_t>(q_abs.size() * 2);
  uint16_t* d_qp = buf.alloc<uint16_t>(q_pe.size() * 2);
  int32_t* d_table = buf.alloc<int32_t>(table.size() * 4);
  int32_t* d_lens = buf.alloc<int32_t>(kB * 4);
  mla_chunk_t* d_chunks = buf.alloc<mla_chunk_t>(N * sizeof(mla_chunk_t));
  int32_t* d_indptr = buf.alloc<int32_t>((kB + 1) * 4);
  float* d_part = buf.alloc<float>(mla_partials_bytes(N, 1, kH));
  float* d_lse = buf.alloc<float>(mla_lse_bytes(N, 1, kH));
  float* d_out = buf.alloc<float>(static_cast<size_t>(kB) * kH * kRank * 4);
  float* d_out_lse = buf.alloc<float>(static_cast<size_t>(kB) * kH * 4);
  const int subs = simt ? 1 : plan.clusters_per_chunk;
  const uint64_t ws_bytes = mla_workspace_bytes(N, subs, plan.cluster_ctas, 1, kH);
  void* d_ws = ws_bytes ? buf.alloc<uint8_t>(ws_bytes) : nullptr;
  if (!d_ckv || !d_kpe || !d_qa || !d_qp || !d_table || !d_lens || !d_chunks || !d_indptr || !d_part || !d_lse ||
      !d_out || !d_out_lse || (ws_bytes && !d_ws))
    return MLA_ERR_CUDA;
  const std::vector<int32_t> lens(kLens, kLens + kB);
  if (!upload(d_ckv, bits(ckv)) || !upload(d_kpe, bits(kpe)) || !upload(d_qa, bits(q_abs)) ||
      !upload(d_qp, bits(q_pe)) || !upload(d_table, table) || !upload(d_lens, lens) || !upload(d_chunks, chunks) ||
      !upload(d_indptr, indptr) || (d_ws && cudaMemset(d_ws, 0, ws_bytes) != cudaSuccess))
    return MLA_ERR_CUDA;

  // decode through the public calls, on a stream of its own
  cudaStream_t s;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return MLA_ERR_CUDA;
  mla_decode_desc_t d;
  std::memset(&d, 0, sizeof(d));
  d.num_requests = kB;
  d.num_heads = kH;
  d.q_len = 1;
  d.block_size = kBs;
  d.num_blocks = kPool;
  d.max_blocks_per_req = max_blocks;
  d.dtype = dtype;
  d.chunks = d_chunks;
  d.num_chunks = N;
  d.cluster_ctas = simt ? 0 : plan.cluster_ctas;
  d.kernel = simt ? MLA_KERNEL_SIMT : MLA_KERNEL_AUTO;
  d.stream = s;
  d.clusters_per_chunk = subs;
  d.workspace = d_ws;
  d.workspace_bytes = ws_bytes;
  st = mla_decode_partial(d_qa, d_qp, d_ckv, d_kpe, d_table, d_lens, kScale, 0, d_part, d_lse, &d);
  if (st == MLA_OK) st = mla_merge_states(d_part, d_lse, d_indptr, kB, 1, kH, d_out, MLA_F32, d_out_lse, s);
  const mla_status_t dev_st = mla_check_device_errors(s, nullptr);  // synchronizes the stream
  cudaStreamDestroy(s);
  if (st != MLA_OK) return st;
  if (dev_st != MLA_OK) return dev_st;
  std::vector<float> out(want.size()), out_lse(want_lse.size());
  if (cudaMemcpy(out.data(), d_out, out.size() * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(out_lse.data(), d_out_lse, out_lse.size() * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MLA_ERR_CUDA;

  // needle rows are exact up to the fp32 division by a sum that rounds to 1; the mean row and
  // the LSEs carry fp32 rounding over a few thousand terms
  double err = 0.0;
  bool ok = true;
  for (int b = 0; b < kB; ++b) {
    for (int h = 0; h < kH; ++h) {
      const size_t o = (static_cast<size_t>(b) * kH + h) * kRank;
      const double tol = h < 15 ? 1e-6 : 2e-3;
      for (int dd = 0; dd < kRank; ++dd) {
        const double e = std::fabs(static_cast<double>(out[o + dd]) - want[o + dd]);
        if (!(e <= tol)) ok = false;
        if (e > err || e != e) err = e != e ? INFINITY : e;
      }
      const double el = std::fabs(static_cast<double>(out_lse[b * kH + h]) - want_lse[b * kH + h]);
      if (!(el <= 1e-3)) ok = false;
    }
  }
  if (max_err != nullptr && static_cast<float>(err) > *max_err) *max_err = static_cast<float>(err);
  return ok ? MLA_OK : MLA_ERR_DEVICE_CHECK;
}

}  // namespace

extern "C" mla_status_t mla_selfcheck(float* max_abs_err) {
  if (max_abs_err != nullptr) *max_abs_err = 0.f;
  for (int dtype : {MLA_F16, MLA_BF16}) {
    for (bool simt : {false, true}) {
      const mla_status_t st = run_one(dtype, simt, max_abs_err);
      if (st != MLA_OK) return st;
    }
  }
  return MLA_OK;
}
