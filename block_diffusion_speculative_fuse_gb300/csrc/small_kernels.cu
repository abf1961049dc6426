// Row-wise and integer kernels of the draft step: block embedding, RMSNorm,
// LM-head argmax reduction, greedy verify and the synthetic target stand-in.
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace dflash {

static std::atomic<uint64_t> g_launches{0};
uint64_t launch_count() { return g_launches.load(); }
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static cudaLaunchAttribute pdl_attr() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

template <typename... KArgs, typename... Args>
static cudaError_t launch(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          bool pdl, Args... args) {
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  count_launch();
  return cudaLaunchKernelEx(&cfg, k, static_cast<KArgs>(args)...);
}

constexpr int kRowThreads = 256;

__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  if (threadIdx.x < 32) {
    t = threadIdx.x < blockDim.x / 32 ? red[threadIdx.x] : 0.f;
    t = warp_sum(t);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  t = red[0];
  __syncthreads();
  return t;
}

// Per-row prologue of a layer stack: x[r] = float(src row), xg[r] =
// bf16(x[r] * g) and ssq[r][t] = sum of x^2 over the 128-column tile t (the
// next GEMM applies 1/rms per row).  Each thread takes 8 consecutive columns
// (one 16-byte load of src and of g, all issued before any is used); the 16
// threads of a tile sum their squares in a fixed order (per thread in column
// order, then a 4-step xor butterfly over the 16 lanes).
__device__ __forceinline__ void row_prologue(const uint16_t* src, const uint16_t* g, int H,
                                             float* x, uint16_t* xg, float* ssq) {
  constexpr int kMaxChunks = 4;  // H <= 8 * kRowThreads * kMaxChunks
  uint4 sv[kMaxChunks], gv[kMaxChunks];
#pragma unroll
  for (int k = 0; k < kMaxChunks; ++k) {
    const int c = (threadIdx.x + k * blockDim.x) * 8;
    if (c < H) {
      sv[k] = __ldg(reinterpret_cast<const uint4*>(src + c));
      gv[k] = __ldg(reinterpret_cast<const uint4*>(g + c));
    }
  }
#pragma unroll
  for (int k = 0; k < kMaxChunks; ++k) {
    const int c = (threadIdx.x + k * blockDim.x) * 8;
    float ss = 0.f;
    if (c < H) {
      const uint16_t* s16 = reinterpret_cast<const uint16_t*>(&sv[k]);
      const uint16_t* g16 = reinterpret_cast<const uint16_t*>(&gv[k]);
      float v[8];
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v[j] = bf2f(s16[j]);
        ss = fmaf(v[j], v[j], ss);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        o[j] = static_cast<uint32_t>(f2bf(v[2 * j] * bf2f(g16[2 * j]))) |
               (static_cast<uint32_t>(f2bf(v[2 * j + 1] * bf2f(g16[2 * j + 1]))) << 16);
      *reinterpret_cast<float4*>(x + c) = make_float4(v[0], v[1], v[2], v[3]);
      *reinterpret_cast<float4*>(x + c + 4) = make_float4(v[4], v[5], v[6], v[7]);
      *reinterpret_cast<uint4*>(xg + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    // the 16 threads of a 128-column tile are 16 consecutive lanes
#pragma unroll
    for (int w = 8; w > 0; w >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, w);
    if (c < H && (threadIdx.x % 16) == 0) ssq[c / 128] = ss;
  }
}

// Block rows: E[anchor] at block position 0, mask_embed at 1..B-1.  Blocks
// past the block rows copy the pending context rows into a[n_blk + t] so the
// first QKV GEMM sees [block rows ; context rows] as one operand.
__global__ void __launch_bounds__(kRowThreads)
    embed_block_kernel(const int32_t* anchor, int block, int n_blk, const uint16_t* embed,
                       const uint16_t* mask_embed, const uint16_t* g, int H, float* x,
                       uint16_t* a, int ld_a, float* ssq, const uint16_t* pending,
                       int32_t* status, int vocab) {
  griddep_launch_dependents();
  griddep_wait();
  const int r = blockIdx.x;
  if (r >= n_blk) {
    const uint4* src = reinterpret_cast<const uint4*>(pending + static_cast<size_t>(r - n_blk) * H);
    uint4* dst = reinterpret_cast<uint4*>(a + static_cast<size_t>(r) * ld_a);
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = threadIdx.x + k * blockDim.x;
      if (i < H / 8) v[k] = __ldcg(src + i);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = threadIdx.x + k * blockDim.x;
      if (i < H / 8) dst[i] = v[k];
    }
    return;
  }
  const int req = r / block, i = r % block;
  const uint16_t* src = mask_embed;
  if (i == 0) {
    int tok = anchor[req];
    if (tok < 0 || tok >= vocab) {
      if (threadIdx.x == 0) raise_status(status, DFLASH_ERR_INVALID_ARG, 301);
      tok = 0;
    }
    src = embed + static_cast<size_t>(tok) * H;
  }
  row_prologue(src, g, H, x + static_cast<size_t>(r) * H, a + static_cast<size_t>(r) * ld_a,
               ssq + static_cast<size_t>(r) * (H / 128));
}

__global__ void __launch_bounds__(kRowThreads)
    embed_tokens_kernel(const int32_t* tokens, const uint16_t* embed, const uint16_t* g, int H,
                        float* x, uint16_t* a, float* ssq, int32_t* status, int vocab) {
  griddep_launch_dependents();
  griddep_wait();
  const int r = blockIdx.x;
  int tok = tokens[r];
  if (tok < 0 || tok >= vocab) {
    if (threadIdx.x == 0) raise_status(status, DFLASH_ERR_INVALID_ARG, 302);
    tok = 0;
  }
  row_prologue(embed + static_cast<size_t>(tok) * H, g, H, x + static_cast<size_t>(r) * H,
               a + static_cast<size_t>(r) * H, ssq + static_cast<size_t>(r) * (H / 128));
}

// out[r] = bf16(x[r] * g / sqrt(mean(x[r]^2) + eps)); raw_out[r] = bf16(x[r]).
__global__ void __launch_bounds__(kRowThreads)
    rmsnorm_kernel(const float* x, int H, const uint16_t* g, float eps, uint16_t* out, int ld_out,
                   uint16_t* raw_out, int ld_raw) {
  __shared__ float red[32];
  griddep_launch_dependents();
  // the gains are not written by any kernel: load them before the wait
  constexpr int kMaxChunks = 4;  // H <= 8 * kRowThreads * kMaxChunks
  uint4 gv[kMaxChunks];
#pragma unroll
  for (int k = 0; k < kMaxChunks; ++k) {
    const int c = (threadIdx.x + k * blockDim.x) * 8;
    if (c < H) gv[k] = __ldg(reinterpret_cast<const uint4*>(g + c));
  }
  griddep_wait();
  const int r = blockIdx.x;
  const float* xr = x + static_cast<size_t>(r) * H;
  // thread t takes columns 8t..8t+7 (+ 8 blockDim for the next chunk): every
  // load in flight at once
  float4 xv[kMaxChunks][2];
#pragma unroll
  for (int k = 0; k < kMaxChunks; ++k) {
    const int c = (threadIdx.x + k * blockDim.x) * 8;
    if (c < H) {
      xv[k][0] = __ldcg(reinterpret_cast<const float4*>(xr + c));
      xv[k][1] = __ldcg(reinterpret_cast<const float4*>(xr + c + 4));
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxChunks; ++k) {
    const int c = (threadIdx.x + k * blockDim.x) * 8;
    if (c < H) {
      const float v[8] = {xv[k][0].x, xv[k][0].y, xv[k][0].z, xv[k][0].w,
                          xv[k][1].x, xv[k][1].y, xv[k][1].z, xv[k][1].w};
#pragma unroll
      for (int j = 0; j < 8; ++j) ss = fmaf(v[j], v[j], ss);
      if (raw_out != nullptr) {
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = pack_bf2(v[2 * j], v[2 * j + 1]);
        *reinterpret_cast<uint4*>(raw_out + static_cast<size_t>(r) * ld_raw + c) =
            make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / static_cast<float>(H) + eps);
#pragma unroll
  for (int k = 0; k < kMaxChunks; ++k) {
    const int c = (threadIdx.x + k * blockDim.x) * 8;
    if (c < H) {
      const float v[8] = {xv[k][0].x, xv[k][0].y, xv[k][0].z, xv[k][0].w,
                          xv[k][1].x, xv[k][1].y, xv[k][1].z, xv[k][1].w};
      const uint16_t* g16 = reinterpret_cast<const uint16_t*>(&gv[k]);
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        o[j] = pack_bf2(v[2 * j] * inv * bf2f(g16[2 * j]), v[2 * j + 1] * inv * bf2f(g16[2 * j + 1]));
      *reinterpret_cast<uint4*>(out + static_cast<size_t>(r) * ld_out + c) =
          make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// One warp per row: (max, lowest index) over the per-tile partials.
__global__ void __launch_bounds__(128)
    argmax_reduce_kernel(const float* val, const int32_t* idx, int rows, int n_tiles, int block,
                         int32_t* out, int skip_first) {
  griddep_launch_dependents();
  griddep_wait();
  const int row = blockIdx.x * 4 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= rows) return;
  const int i = row % block;
  if (skip_first && i == 0) return;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int t = lane; t < n_tiles; t += 32) {
    const float v = val[static_cast<size_t>(row) * n_tiles + t];
    const int j = idx[static_cast<size_t>(row) * n_tiles + t];
    if (v > bv || (v == bv && j < bi)) { bv = v; bi = j; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
  }
  if (lane == 0) {
    if (skip_first)
      out[(row / block) * (block - 1) + i - 1] = bi;
    else
      out[row] = bi;
  }
}

// One warp per request: ballot of mismatches, n = index of the first one.
__global__ void __launch_bounds__(128)
    verify_kernel(const int32_t* draft, const int32_t* target, int batch, int B,
                  int32_t* out_tokens, int32_t* n_accept, const int32_t* tgt_len_in,
                  int32_t* tgt_len_out, int32_t* ctx_pending, int32_t* anchor_out,
                  const int32_t* anchor_pos_in, int32_t* anchor_pos_out, int32_t* ctx_pos) {
  griddep_launch_dependents();
  griddep_wait();
  const int r = blockIdx.x * 4 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (r >= batch) return;
  const int t = lane < B ? target[static_cast<size_t>(r) * B + lane] : 0;
  const bool mism = lane < B - 1 && draft[static_cast<size_t>(r) * (B - 1) + lane] != t;
  const unsigned mask = __ballot_sync(0xffffffffu, mism);
  const int n = mask ? __ffs(mask) - 1 : B - 1;
  const int bonus = __shfl_sync(0xffffffffu, t, n);
  const int tl = (lane == 0 && tgt_len_in != nullptr) ? tgt_len_in[r] : 0;
  const int ap = __shfl_sync(0xffffffffu, (lane == 0 && anchor_pos_in != nullptr) ? anchor_pos_in[r] : 0, 0);
  __syncwarp();
  if (lane < B && out_tokens != nullptr)
    out_tokens[static_cast<size_t>(r) * B + lane] = lane <= n ? t : -1;
  if (lane < B && ctx_pos != nullptr) ctx_pos[static_cast<size_t>(r) * B + lane] = lane <= n ? ap + lane : -1;
  if (lane == 0) {
    if (n_accept != nullptr) n_accept[r] = n;
    if (tgt_len_out != nullptr) tgt_len_out[r] = tl + n + 1;
    if (ctx_pending != nullptr) ctx_pending[r] = n + 1;
    if (anchor_out != nullptr) anchor_out[r] = bonus;
    if (anchor_pos_out != nullptr) anchor_pos_out[r] = ap + n + 1;
  }
}

// ---- E4M3 context cache: one warp per cached vector (position, K|V, head)
// of d bf16 values: scale = amax / 448 (1 for a zero vector), codes of
// value / scale rounded to nearest, ties to even, saturating.
__global__ void __launch_bounds__(256)
    kv_quantize_kernel(const uint16_t* src, uint8_t* dst, float* scales, size_t vectors, int d) {
  griddep_launch_dependents();
  griddep_wait();
  const size_t vec = static_cast<size_t>(blockIdx.x) * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (vec >= vectors) return;
  const int per = d / 32;  // 2 or 4 values per lane
  const uint16_t* s = src + vec * d + lane * per;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < per; ++j) v[j] = bf2f(s[j]);
  float a = 0.f;
  for (int j = 0; j < per; ++j) a = fmaxf(a, fabsf(v[j]));
  a = warp_max(a);
  const float scale = a > 0.f ? a / 448.f : 1.f;
  uint8_t* o = dst + vec * d + lane * per;
  if (per == 4) {
    const uint32_t c = static_cast<uint32_t>(e4m3x2_encode(v[0] / scale, v[1] / scale)) |
                       (static_cast<uint32_t>(e4m3x2_encode(v[2] / scale, v[3] / scale)) << 16);
    *reinterpret_cast<uint32_t*>(o) = c;
  } else {
    *reinterpret_cast<uint16_t*>(o) = e4m3x2_encode(v[0] / scale, v[1] / scale);
  }
  if (lane == 0) scales[vec] = scale;
}

// ---- synthetic target (counter-based, splitmix64 output function)
__device__ __forceinline__ uint64_t splitmix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
__device__ __forceinline__ uint64_t synth_key(uint64_t seed, uint64_t step, uint64_t r, uint64_t i,
                                              uint64_t stream) {
  constexpr uint64_t M = 0x100000001B3ull;
  uint64_t k = seed;
  k = k * M + step;
  k = k * M + r;
  k = k * M + i;
  k = k * M + stream;
  return k;
}

__global__ void synth_target_kernel(const int32_t* draft, int batch, int B, const uint64_t* thr,
                                    int vocab, uint64_t seed, int64_t* step, int advance,
                                    int32_t* target) {
  griddep_launch_dependents();
  griddep_wait();
  const uint64_t st = static_cast<uint64_t>(*step);
  __syncthreads();
  for (int idx = threadIdx.x; idx < batch * B; idx += blockDim.x) {
    const int r = idx / B, i = idx % B;
    const uint64_t h0 = splitmix64(synth_key(seed, st, r, i, 0));
    const uint64_t h1 = splitmix64(synth_key(seed, st, r, i, 1));
    int32_t t;
    if (i < B - 1) {
      const int32_t d = draft[static_cast<size_t>(r) * (B - 1) + i];
      if ((h0 >> 11) < thr[r])
        t = d;
      else
        t = static_cast<int32_t>((static_cast<uint64_t>(d) + 1 + h1 % static_cast<uint64_t>(vocab - 1)) %
                                 static_cast<uint64_t>(vocab));
    } else {
      t = static_cast<int32_t>(h1 % static_cast<uint64_t>(vocab));
    }
    target[idx] = t;
  }
  __syncthreads();
  if (threadIdx.x == 0 && advance) *step = static_cast<int64_t>(st + 1);
}

__global__ void copy_f32_kernel(const float* src, float* dst, size_t n) {
  griddep_launch_dependents();
  griddep_wait();
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    dst[i] = src[i];
}

// ---------------------------------------------------------------- launchers
cudaError_t embed_block_launch(const int32_t* anchor, int batch, int block, const uint16_t* embed,
                               const uint16_t* mask_embed, const uint16_t* norm, int hidden,
                               float* x, uint16_t* a, int ld_a, float* ssq,
                               const uint16_t* pending, int T, cudaStream_t s, bool pdl,
                               int32_t* status, int vocab) {
  const int nb = batch * block;
  return launch(embed_block_kernel, dim3(nb + T), dim3(kRowThreads), 0, s, pdl, anchor, block, nb,
                embed, mask_embed, norm, hidden, x, a, ld_a, ssq, pending, status, vocab);
}
cudaError_t embed_tokens_launch(const int32_t* tokens, int rows, const uint16_t* embed,
                                const uint16_t* norm, int hidden, float* x, uint16_t* a,
                                float* ssq, cudaStream_t s, bool pdl, int32_t* status,
                                int vocab) {
  return launch(embed_tokens_kernel, dim3(rows), dim3(kRowThreads), 0, s, pdl, tokens, embed, norm,
                hidden, x, a, ssq, status, vocab);
}
cudaError_t rmsnorm_launch(const float* x, int rows, int hidden, const uint16_t* g, float eps,
                           uint16_t* out, int ld_out, uint16_t* raw_out, int ld_raw,
                           cudaStream_t s, bool pdl) {
  return launch(rmsnorm_kernel, dim3(rows), dim3(kRowThreads), 0, s, pdl, x, hidden, g, eps, out,
                ld_out, raw_out, ld_raw);
}
cudaError_t argmax_reduce_launch(const float* val, const int32_t* idx, int rows, int n_tiles,
                                 int block, int32_t* out, int skip_first, cudaStream_t s,
                                 bool pdl) {
  return launch(argmax_reduce_kernel, dim3((rows + 3) / 4), dim3(128), 0, s, pdl, val, idx, rows,
                n_tiles, block, out, skip_first);
}
cudaError_t kv_quantize_launch(const uint16_t* src, uint8_t* dst, float* scales, size_t vectors,
                               int d, cudaStream_t s, bool pdl) {
  const size_t blocks = (vectors + 7) / 8;
  if (blocks == 0 || blocks > 0x7FFFFFFFu) return cudaErrorInvalidValue;
  return launch(kv_quantize_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, pdl, src,
                dst, scales, vectors, d);
}
cudaError_t verify_launch(const int32_t* draft, const int32_t* target, int batch, int B,
                          int32_t* out_tokens, int32_t* n_accept, const int32_t* tgt_len_in,
                          int32_t* tgt_len_out, int32_t* ctx_pending, int32_t* anchor_out,
                          const int32_t* anchor_pos_in, int32_t* anchor_pos_out, int32_t* ctx_pos,
                          cudaStream_t s, bool pdl) {
  return launch(verify_kernel, dim3((batch + 3) / 4), dim3(128), 0, s, pdl, draft, target, batch,
                B, out_tokens, n_accept, tgt_len_in, tgt_len_out, ctx_pending, anchor_out,
                anchor_pos_in, anchor_pos_out, ctx_pos);
}
cudaError_t synth_target_launch(const int32_t* draft, int batch, int B, const uint64_t* thr,
                                int vocab, uint64_t seed, int64_t* step, int advance,
                                int32_t* target, cudaStream_t s, bool pdl) {
  return launch(synth_target_kernel, dim3(1), dim3(1024), 0, s, pdl, draft, batch, B, thr, vocab,
                seed, step, advance, target);
}
// Self-test of the path every bounded wait takes when it runs out: thread 0
// initialises an mbarrier in its own shared memory for one arrival, arrives
// on it only when `arrive` is set, then waits for phase 0 for at most
// limit_ns.  A wait that gives up records DFLASH_ERR_TIMEOUT (site 901) and
// the kernel returns as usual.  No copy is ever issued on the barrier, so
// nothing is left in flight when the kernel exits.
__global__ void wait_selftest_kernel(int arrive, uint64_t limit_ns, int* status,
                                     int64_t* waited_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_barrier_init();
  if (arrive) mbar_arrive(&bar);
  const uint64_t t0 = global_ns();
  const bool ok = mbar_wait_for(&bar, 0, nullptr, limit_ns);
  const uint64_t t1 = global_ns();
  if (!ok) raise_status(status, DFLASH_ERR_TIMEOUT, 901);
  if (waited_ns != nullptr) *waited_ns = static_cast<int64_t>(t1 - t0);
}

cudaError_t wait_selftest_launch(int arrive, uint64_t limit_ns, int* status, int64_t* waited_ns,
                                 cudaStream_t s) {
  return launch(wait_selftest_kernel, dim3(1), dim3(32), 0, s, false, arrive, limit_ns, status,
                waited_ns);
}
cudaError_t copy_rows_f32_launch(const float* src, float* dst, size_t n, cudaStream_t s, bool pdl) {
  const int blocks = static_cast<int>((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
  return launch(copy_f32_kernel, dim3(blocks > 0 ? blocks : 1), dim3(256), 0, s, pdl, src, dst, n);
}

}  // namespace dflash
