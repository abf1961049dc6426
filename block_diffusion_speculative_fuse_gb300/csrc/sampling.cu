// Speculative verification at temperature T > 0, and draft sampling.
//
// The rule is the standard lossless one of speculative sampling, applied per
// block position (the drafter's q_i for every position comes out of one
// parallel pass, so each d_i ~ q_i is drawn independently):
//   q_i = softmax(z_i / T), p_j = softmax(y_j / T);
//   accept d_i when u_i q_i(d_i) < p_i(d_i); at the first rejection emit a
//   draw from max(0, p_i - q_i); after B-1 acceptances a bonus draw from p_B.
// Every draw is an inverse-CDF draw with a uniform a passed in: the smallest
// k with a * S < C_k (C_k the running sum of the weights, S their total).
//
// Arithmetic: row maxima in fp32 (exact), exponentials of (z - max) / T in
// fp32; the row statistics and the draws from a softmax (draft sampling,
// the bonus token) add each thread's exponentials in fp32 with Kahan
// compensation and combine the thread sums in fp64 (the GPU's fp64 rate is
// low, and a plain fp64 sum per element set the pace); the residual draw
// max(0, p - q) sums in fp64 (its terms cancel); every running sum over the
// threads is fp64, in a fixed order; the accept test evaluates its two
// probabilities with fp64 exp.  Against an all-fp64 evaluation a decision
// can therefore differ only when its uniform lies within about 1e-6
// (relative) of a boundary.
//
// Kernels:
//   sample_stats_kernel   one CTA per logits row: (max, S) of the row
//   verify_sampling_kernel one CTA per request: accept loop, then the
//                          residual (or bonus) draw over the vocabulary
//   sample_rows_kernel    one CTA per row: categorical draw from softmax(z/T)
#include "common.cuh"
#include "kernels.h"

namespace dflash {

namespace {

constexpr int kSampThreads = 1024;
constexpr int kSampWarps = kSampThreads / 32;

__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Fixed-order block sum (warp butterflies, then the warp sums in order).
__device__ double block_sum_f64(double v, double* red) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  v = warp_sum_f64(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  double t = 0.0;
  if (warp == 0) {
    t = lane < kSampWarps ? red[lane] : 0.0;
    t = warp_sum_f64(t);
    if (lane == 0) red[0] = t;
  }
  __syncthreads();
  t = red[0];
  __syncthreads();
  return t;
}

__device__ float block_max_f32(float v, float* red) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  v = warp_max(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float t = lane < kSampWarps ? red[lane] : -INFINITY;
    t = warp_max(t);
    if (lane == 0) red[0] = t;
  }
  __syncthreads();
  const float t = red[0];
  __syncthreads();
  return t;
}

// Exclusive prefix of one fp64 value per thread in thread order (a
// Hillis-Steele scan over the warp sums, then within each warp).
__device__ double block_exclusive_scan_f64(double v, double* red, double* total) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  double incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) red[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    double w = lane < kSampWarps ? red[lane] : 0.0;
    double wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    red[32 + lane] = wi - w;  // exclusive prefix of the warp sums
    if (lane == 31) red[64] = wi;
  }
  __syncthreads();
  const double ex = red[32 + warp] + (incl - v);
  *total = red[64];
  __syncthreads();
  return ex;
}

// Inverse-CDF draw over V weights given by wfn(k) >= 0 (fp64): thread t takes
// the contiguous segment [t*seg, (t+1)*seg); the segment sums are scanned in
// thread order and the thread whose segment holds a*S walks it.  Returns the
// index on every thread (V-1 if rounding leaves a*S at or past the total).
template <typename WFn>
__device__ int draw_inverse_cdf(int V, double a, WFn wfn, double* red, int* found) {
  const int seg = (V + kSampThreads - 1) / kSampThreads;
  const int k0 = threadIdx.x * seg, k1 = min(V, k0 + seg);
  double s = 0.0;
  for (int k = k0; k < k1; ++k) s += wfn(k);
  double S = 0.0;
  const double pre = block_exclusive_scan_f64(s, red, &S);
  const double target = a * S;
  if (threadIdx.x == 0) *found = V - 1;
  __syncthreads();
  if (pre <= target && target < pre + s) {
    double c = pre;
    int k = k1 - 1;
    for (int j = k0; j < k1; ++j) {
      c += wfn(j);
      if (target < c) {
        k = j;
        break;
      }
    }
    atomicMin(found, k);
  }
  __syncthreads();
  const int k = *found;
  __syncthreads();
  return k;
}

// The same draw for weights given in fp32 by wfn(k) >= 0 with no
// cancellation in them (exponentials): each thread's segment sum in fp32
// with Kahan compensation, the scan of the segment sums and the walk in
// fp64.  The walk adds the same terms in fp64, so a target within a few fp32
// ulps of a segment's end can fall past its last element; the draw then
// returns that element.
template <typename WFn>
__device__ int draw_inverse_cdf_f32(int V, double a, WFn wfn, double* red, int* found) {
  const int seg = (V + kSampThreads - 1) / kSampThreads;
  const int k0 = threadIdx.x * seg, k1 = min(V, k0 + seg);
  float s = 0.f, comp = 0.f;
  for (int k = k0; k < k1; ++k) {
    const float y = wfn(k) - comp;
    const float t = s + y;
    comp = (t - s) - y;
    s = t;
  }
  const double sd = static_cast<double>(s) - static_cast<double>(comp);
  double S = 0.0;
  const double pre = block_exclusive_scan_f64(sd, red, &S);
  const double target = a * S;
  if (threadIdx.x == 0) *found = V - 1;
  __syncthreads();
  if (k0 < k1 && pre <= target && target < pre + sd) {
    double c = pre;
    int k = k1 - 1;
    for (int j = k0; j < k1; ++j) {
      c += static_cast<double>(wfn(j));
      if (target < c) {
        k = j;
        break;
      }
    }
    atomicMin(found, k);
  }
  __syncthreads();
  const int k = *found;
  __syncthreads();
  return k;
}
// Row rr of a blocked logits array [.][block][V] whose first `skip` rows of
// every block are not used: block rr / (block - skip), row skip + rr % (...).
__device__ __forceinline__ const float* blocked_row(const float* base, int rr, int block, int skip,
                                                    int V) {
  const int per = block - skip;
  return base + (static_cast<size_t>(rr / per) * block + skip + rr % per) * V;
}

// (max, S) of each logits row: the nq used rows of the blocked array q_rows
// (block q_block, first q_skip rows of each block unused), then np rows of
// p_rows, each V floats.  stats[r] = (max, sum of exp((z - max) / T)).
__global__ void __launch_bounds__(kSampThreads)
    sample_stats_kernel(const float* q_rows, int nq, int q_block, int q_skip, const float* p_rows,
                        int np, int V, float T, double2* stats) {
  __shared__ float redf[32];
  __shared__ double redd[32];
  griddep_launch_dependents();
  griddep_wait();
  const int r = blockIdx.x;
  if (r >= nq + np) return;
  const float* z = r < nq ? blocked_row(q_rows, r, q_block, q_skip, V)
                          : p_rows + static_cast<size_t>(r - nq) * V;
  const bool vec = V % 4 == 0 && (reinterpret_cast<uintptr_t>(z) & 15) == 0;
  const float4* z4 = reinterpret_cast<const float4*>(z);
  float mx = -INFINITY;
  if (vec) {
    for (int k = threadIdx.x; k < V / 4; k += kSampThreads) {
      const float4 v = __ldg(z4 + k);
      mx = fmaxf(mx, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
    }
  } else {
    for (int k = threadIdx.x; k < V; k += kSampThreads) mx = fmaxf(mx, __ldg(z + k));
  }
  mx = block_max_f32(mx, redf);
  // Each thread adds its exponentials in fp32 with a compensation term
  // (Kahan): the lost low parts are carried, so the thread's sum is within
  // a few fp32 ulps of the exact sum of its terms; the thread sums are then
  // added in fp64 in a fixed order.
  float s = 0.f, comp = 0.f;
  auto add = [&](float x) {
    const float y = expf((x - mx) / T) - comp;
    const float t = s + y;
    comp = (t - s) - y;
    s = t;
  };
  if (vec) {
    for (int k = threadIdx.x; k < V / 4; k += kSampThreads) {
      const float4 v = __ldg(z4 + k);
      add(v.x);
      add(v.y);
      add(v.z);
      add(v.w);
    }
  } else {
    for (int k = threadIdx.x; k < V; k += kSampThreads) add(__ldg(z + k));
  }
  const double S = block_sum_f64(static_cast<double>(s) - static_cast<double>(comp), redd);
  if (threadIdx.x == 0) stats[r] = make_double2(static_cast<double>(mx), S);
}

// Probability of token k in a row with stats (max, S), in fp64.
__device__ __forceinline__ double prob_f64(const float* z, int k, double2 st, double T) {
  return exp((static_cast<double>(z[k]) - st.x) / T) / st.y;
}

// q_rows: the drafter's logits [batch][B][V] (block row 0, the anchor, unused:
// row i+1 gives q for draft i); p_rows: the target's [batch][B][V].
__global__ void __launch_bounds__(kSampThreads)
    verify_sampling_kernel(const int32_t* draft, const float* q_rows, const float* p_rows, int B,
                           int V, float T, double Td, const double2* stats, const double* u,
                           const double* w, int32_t* out_tokens, int32_t* n_accept,
                           const int32_t* tgt_len_in, int32_t* tgt_len_out, int32_t* ctx_pending,
                           int32_t* anchor_out, const int32_t* anchor_pos_in,
                           int32_t* anchor_pos_out, int32_t* ctx_pos, int batch,
                           int32_t* status) {
  __shared__ double red[72];
  __shared__ int found;
  __shared__ int s_n;
  griddep_launch_dependents();
  griddep_wait();
  const int r = blockIdx.x;
  const int Bm1 = B - 1;
  const int nq = batch * Bm1;
  const float* zq = q_rows + (static_cast<size_t>(r) * B + 1) * V;  // q rows of this request
  const float* yp = p_rows + static_cast<size_t>(r) * B * V;        // p rows of this request
  // accept loop: one thread, two fp64 probabilities per position
  if (threadIdx.x == 0) {
    int i = 0;
    for (; i < Bm1; ++i) {
      const int d = draft[static_cast<size_t>(r) * Bm1 + i];
      if (d < 0 || d >= V) {
        raise_status(status, DFLASH_ERR_INVALID_ARG, 401);
        break;  // an invalid draft token is rejected
      }
      const double qd = prob_f64(zq + static_cast<size_t>(i) * V, d, stats[r * Bm1 + i], Td);
      const double pd = prob_f64(yp + static_cast<size_t>(i) * V, d, stats[nq + r * B + i], Td);
      if (!(u[static_cast<size_t>(r) * Bm1 + i] * qd < pd)) break;
      out_tokens[static_cast<size_t>(r) * B + i] = d;
    }
    s_n = i;
  }
  __syncthreads();
  const int n = s_n;
  // the emitted target token: residual max(0, p - q) at the first rejection,
  // or the bonus from p_B
  const double a = w[static_cast<size_t>(r) * B + n];
  const float* prow = yp + static_cast<size_t>(n) * V;
  const double2 sp = stats[nq + r * B + n];
  const float mp = static_cast<float>(sp.x);
  const double ip = 1.0 / sp.y;
  int tok;
  if (n < Bm1) {
    const float* qrow = zq + static_cast<size_t>(n) * V;
    const double2 sq = stats[r * Bm1 + n];
    const float mq = static_cast<float>(sq.x);
    const double iq = 1.0 / sq.y;
    tok = draw_inverse_cdf(V, a, [&](int k) {
      const double pk = static_cast<double>(expf((__ldg(prow + k) - mp) / T)) * ip;
      const double qk = static_cast<double>(expf((__ldg(qrow + k) - mq) / T)) * iq;
      return pk > qk ? pk - qk : 0.0;
    }, red, &found);
  } else {
    tok = draw_inverse_cdf_f32(V, a, [&](int k) { return expf((__ldg(prow + k) - mp) / T); }, red,
                               &found);
  }
  if (threadIdx.x < B) {
    const int j = threadIdx.x;
    if (j == n) out_tokens[static_cast<size_t>(r) * B + j] = tok;
    if (j > n) out_tokens[static_cast<size_t>(r) * B + j] = -1;
    if (ctx_pos != nullptr) ctx_pos[static_cast<size_t>(r) * B + j] = j <= n ? anchor_pos_in[r] + j : -1;
  }
  if (threadIdx.x == 0) {
    if (n_accept != nullptr) n_accept[r] = n;
    if (tgt_len_out != nullptr) tgt_len_out[r] = tgt_len_in[r] + n + 1;
    if (ctx_pending != nullptr) ctx_pending[r] = n + 1;
    if (anchor_out != nullptr) anchor_out[r] = tok;
    if (anchor_pos_out != nullptr) anchor_pos_out[r] = anchor_pos_in[r] + n + 1;
  }
}

// One categorical draw per used row of a blocked logits array from
// softmax(z / T) (row stats precomputed): out[r] for used row r.
__global__ void __launch_bounds__(kSampThreads)
    sample_rows_kernel(const float* rows, int block, int skip, int V, float T,
                       const double2* stats, const double* a, int32_t* out) {
  __shared__ double red[72];
  __shared__ int found;
  griddep_launch_dependents();
  griddep_wait();
  const int r = blockIdx.x;
  const float* z = blocked_row(rows, r, block, skip, V);
  const float m = static_cast<float>(stats[r].x);
  const int k = draw_inverse_cdf_f32(V, a[r], [&](int j) { return expf((__ldg(z + j) - m) / T); },
                                     red, &found);
  if (threadIdx.x == 0) out[r] = k;
}

cudaError_t launch_k(const void* fn, dim3 grid, void** args, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kSampThreads, 1, 1);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  count_launch();
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

cudaError_t verify_sampling_launch(const int32_t* draft, const float* q_rows, const float* p_rows,
                                   int batch, int B, int V, double T, const double* u,
                                   const double* w, double2* stats, int32_t* out_tokens,
                                   int32_t* n_accept, const int32_t* tgt_len_in,
                                   int32_t* tgt_len_out, int32_t* ctx_pending,
                                   int32_t* anchor_out, const int32_t* anchor_pos_in,
                                   int32_t* anchor_pos_out, int32_t* ctx_pos, int32_t* status,
                                   cudaStream_t s, bool pdl) {
  int nq = batch * (B - 1), np = batch * B, one = 1;
  float Tf = static_cast<float>(T);
  void* a1[] = {&q_rows, &nq, &B, &one, &p_rows, &np, &V, &Tf, &stats};
  cudaError_t e = launch_k(reinterpret_cast<const void*>(sample_stats_kernel), dim3(nq + np), a1, s, pdl);
  if (e != cudaSuccess) return e;
  void* a2[] = {&draft, &q_rows, &p_rows, &B, &V, &Tf, &T, &stats, &u, &w, &out_tokens, &n_accept,
                &tgt_len_in, &tgt_len_out, &ctx_pending, &anchor_out, &anchor_pos_in,
                &anchor_pos_out, &ctx_pos, &batch, &status};
  return launch_k(reinterpret_cast<const void*>(verify_sampling_kernel), dim3(batch), a2, s, pdl);
}

cudaError_t sample_rows_launch(const float* rows, int n_used, int block, int skip, int V, double T,
                               const double* a, double2* stats, int32_t* out, cudaStream_t s,
                               bool pdl) {
  const float* none = nullptr;
  int zero = 0;
  float Tf = static_cast<float>(T);
  void* a1[] = {&rows, &n_used, &block, &skip, &none, &zero, &V, &Tf, &stats};
  cudaError_t e = launch_k(reinterpret_cast<const void*>(sample_stats_kernel), dim3(n_used), a1, s, pdl);
  if (e != cudaSuccess) return e;
  void* a2[] = {&rows, &block, &skip, &V, &Tf, &stats, &a, &out};
  return launch_k(reinterpret_cast<const void*>(sample_rows_kernel), dim3(n_used), a2, s, pdl);
}

}  // namespace dflash
