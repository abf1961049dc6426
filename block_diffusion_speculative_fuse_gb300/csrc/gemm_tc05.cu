// Weight-streaming GEMM on the 5th-generation tensor cores (tcgen05, sm_103a).
//
//   Y[m][n] = sum_k X[m][k] * W[n][k]        (y = x W^T, W stored [out][in])
//
// "Swap-AB" orientation: 128 weight rows form the MMA M side, the (few)
// activation rows the MMA N side (BN = 16..256), so a decode-sized batch
// still fills the 128-lane tensor core and the kernel streams W at HBM speed.
//
// Per CTA (128 threads): one 128-row weight tile x one BN-row activation tile
// over a K range (split-K).  Warp 0 lane 0 issues TMA loads into a STAGES-deep
// shared-memory ring (128-byte swizzle, 64 K-elements per stage); warp 1 owns
// the TMEM accumulator and lane 0 issues tcgen05.mma (M=128, N=BN, K=16, four
// per stage), committing each stage back to the producer through an mbarrier.
// With split-K, every CTA writes its fp32 partial tile and the last CTA of a
// tile (atomic ticket, no spinning) sums the partials in split order, so the
// result is deterministic and independent of M.  The final tile is staged in
// shared memory and handed to one of the fused epilogues (bf16/f32 store,
// residual add + DFlash-2 block conv, SwiGLU, q/k-norm + RoPE + KV routing,
// per-tile argmax for the LM head).
//
// Weight loads are issued before griddepcontrol.wait, so with programmatic
// dependent launch a GEMM prefetches its first stages of weights while the
// previous kernel is still draining.
#include "common.cuh"
#include "kernels.h"

namespace dflash {

template <int BN>
struct GemmCfg {
  // BN <= 32 (decode-sized M): 3 CTAs fit per SM, so while a GEMM runs on two
  // slots the next kernel's CTAs (programmatic dependent launch) occupy the
  // third and prefetch their first weight stages.
  static constexpr int STAGES = BN <= 16 ? 4 : BN <= 32 ? 3 : BN <= 64 ? 4 : BN <= 128 ? 6 : 4;
  static constexpr int A_BYTES = kTileN * kTileK * 2;  // 16 KB
  static constexpr int B_BYTES = BN * kTileK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TS_LD = kTileN + 4;  // staged epilogue tile row stride (floats)
  static constexpr int TILE_BYTES = BN * TS_LD * 4;
  static constexpr int PIPE_BYTES = STAGES * STAGE_BYTES;
  static constexpr int MAIN_BYTES = PIPE_BYTES > TILE_BYTES ? PIPE_BYTES : TILE_BYTES;
  // epilogue scratch (row scales, QKV routing) sits after the staged tile
  static constexpr int SCRATCH_OFF = (TILE_BYTES + 255) / 256 * 256;
  static_assert(SCRATCH_OFF + 4 * BN * 4 <= MAIN_BYTES, "epilogue scratch must fit the pipeline region");
  static constexpr int SMEM_BYTES = MAIN_BYTES + 256 + 1024;  // + barriers, alignment slack
  static constexpr int TMEM_COLS = BN < 32 ? 32 : BN;
};

// ---------------------------------------------------------------- RoPE angle
// sin/cos of pos * inv_freq with inv_freq held as an unevaluated float pair
// (hi + lo).  The product is formed exactly with an FMA (Dekker's two-product)
// and reduced modulo 2*pi with a three-piece Cody-Waite split of 2*pi, so the
// reduced angle is accurate to ~1e-6 rad for positions up to 2^24.
__device__ __forceinline__ void rope_sincos(int pos, float2 f, float* s, float* c) {
  const float pf = static_cast<float>(pos);
  const float a_hi = pf * f.x;
  const float a_err = fmaf(pf, f.x, -a_hi);
  const float a_lo = fmaf(pf, f.y, a_err);
  // 2*pi = P1 + P2 + P3 (P1, P2 with trailing zero bits)
  constexpr float P1 = 6.28125f;
  constexpr float P2 = 1.93500518798828125e-3f;
  constexpr float P3 = 3.019916050561733e-07f;
  constexpr float INV_2PI = 0.15915494309189535f;
  const float k = rintf(a_hi * INV_2PI);
  float r = fmaf(-k, P1, a_hi);
  r = fmaf(-k, P2, r);
  r = fmaf(-k, P3, r);
  r += a_lo;
  sincosf(r, s, c);
}

// ---------------------------------------------------------------- epilogues
template <int BN>
__device__ void epi_store(const GemmParams& p, const float* ts, int tile, int m0, int rows) {
  using C = GemmCfg<BN>;
  const int n0 = tile * kTileN;
  for (int idx = threadIdx.x; idx < rows * kTileN; idx += 128) {
    const int r = idx / kTileN, f = idx % kTileN;
    const float v = ts[r * C::TS_LD + f];
    const size_t o = static_cast<size_t>(m0 + r) * p.ld_out + n0 + f;
    if (p.mode == EPI_STORE_BF16)
      static_cast<uint16_t*>(p.out)[o] = f2bf(v);
    else
      static_cast<float*>(p.out)[o] = v;
  }
}

template <int BN>
__device__ void epi_resid(const GemmParams& p, float* ts, int tile, int m0, int rows) {
  using C = GemmCfg<BN>;
  // Thread f owns feature column n0 + f: x_new = x + acc, then the optional
  // depthwise conv along block positions (sliding window down the column,
  // zero padded at each request's block edges), then the next norm's inputs.
  const int f = threadIdx.x;
  const int n = tile * kTileN + f;
  for (int r0 = 0; r0 < rows; r0 += 16) {
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      v[j] = (r0 + j < rows) ? __ldcg(p.resid + static_cast<size_t>(m0 + r0 + j) * p.ld_resid + n) : 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (r0 + j < rows) ts[(r0 + j) * C::TS_LD + f] += v[j];
  }
  if (p.conv != nullptr && p.conv_width > 0) {
    const int c = (p.conv_width - 1) / 2;
    float w[7];
#pragma unroll
    for (int j = 0; j < 7; ++j) w[j] = j < p.conv_width ? bf2f(p.conv[static_cast<size_t>(n) * p.conv_width + j]) : 0.f;
    for (int r0 = 0; r0 < rows; r0 += p.block) {
      float win[7];  // original values x_{i-c} .. x_{i+c} of the current position
#pragma unroll
      for (int j = 0; j < 7; ++j) {
        const int src = j - c;
        win[j] = (j < p.conv_width && src >= 0 && src < p.block) ? ts[(r0 + src) * C::TS_LD + f] : 0.f;
      }
      for (int i = 0; i < p.block; ++i) {
        float y = win[c];
#pragma unroll
        for (int j = 0; j < 7; ++j)
          if (j < p.conv_width) y = fmaf(w[j], win[j], y);
        // slide: drop win[0], append x_{i+1+c}
#pragma unroll
        for (int j = 0; j < 6; ++j) win[j] = win[j + 1];
        const int nxt = i + 1 + c;
        if (p.conv_width > 0) {
          const float v = (nxt < p.block) ? ts[(r0 + nxt) * C::TS_LD + f] : 0.f;
          // window length is conv_width; keep the slot after the last live one
          win[p.conv_width - 1] = v;
        }
        ts[(r0 + i) * C::TS_LD + f] = y;
      }
    }
  }
  for (int r = 0; r < rows; ++r) {
    const float x = ts[r * C::TS_LD + f];
    const size_t m = static_cast<size_t>(m0 + r);
    p.resid[m * p.ld_resid + n] = x;
    if (p.xg_out != nullptr) p.xg_out[m * p.ld_xg + n] = f2bf(x * bf2f(p.gnext[n]));
    if (p.raw_out != nullptr) p.raw_out[m * p.ld_raw + n] = f2bf(x);
  }
  if (p.ssq_out != nullptr) {
    __syncthreads();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    for (int r = warp; r < rows; r += 4) {
      float ss = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float v = ts[r * C::TS_LD + lane + 32 * k];
        ss = fmaf(v, v, ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) p.ssq_out[static_cast<size_t>(m0 + r) * p.ssq_ld + tile] = ss;
    }
  }
}

template <int BN>
__device__ void epi_swiglu(const GemmParams& p, const float* ts, int tile, int m0, int rows) {
  using C = GemmCfg<BN>;
  uint16_t* out = static_cast<uint16_t*>(p.out);
  for (int idx = threadIdx.x; idx < rows * 64; idx += 128) {
    const int r = idx / 64, j = idx % 64;
    const float g = ts[r * C::TS_LD + j];
    const float u = ts[r * C::TS_LD + 64 + j];
    out[static_cast<size_t>(m0 + r) * p.ld_out + tile * 64 + j] = f2bf(silu_f(g) * u);
  }
}

template <int BN>
__device__ void epi_argmax(const GemmParams& p, const float* ts, int tile, int m0, int rows) {
  using C = GemmCfg<BN>;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_tiles = gridDim.x;
  const int n0 = tile * kTileN;
  for (int r = warp; r < rows; r += 4) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int f = lane + 32 * t;
      const float v = ts[r * C::TS_LD + f];
      if (v > bv) { bv = v; bi = n0 + f; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    if (lane == 0) {
      p.amax_val[static_cast<size_t>(m0 + r) * n_tiles + tile] = bv;
      p.amax_idx[static_cast<size_t>(m0 + r) * n_tiles + tile] = bi;
    }
  }
  if (p.logits != nullptr) {
    for (int idx = threadIdx.x; idx < rows * kTileN; idx += 128) {
      const int r = idx / kTileN, f = idx % kTileN;
      p.logits[static_cast<size_t>(m0 + r) * p.ld_logits + n0 + f] = ts[r * C::TS_LD + f];
    }
  }
}

template <int BN>
__device__ void epi_qkv(const GemmParams& p, const float* ts, int tile, int m0, int rows,
                        int* route) {
  using C = GemmCfg<BN>;
  const QkvEpi& e = p.qkv;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int d = e.head_dim;
  const int half = d / 2;
  const int per_tile = kTileN / d;
  const int npair = half / 32;  // pairs per lane: 1 (d=64) or 2 (d=128)
  const int hq = e.n_q_heads, hkv = e.n_kv_heads;
  // Per-row routing, one thread per row, all lookups issued in parallel:
  // route[r] = (request, position, physical page or -1 for block rows / -2 skip)
  int* r_req = route;
  int* r_pos = route + BN;
  int* r_pg = route + 2 * BN;
  for (int r = threadIdx.x; r < rows; r += 128) {
    const int m = m0 + r;
    int req, pos, pg = -1;
    if (m < e.n_blk) {
      req = m / e.block;
      pos = e.anchor_pos[req] + m % e.block;
    } else {
      const int j = m - e.n_blk;
      if (e.pool_req != nullptr) {
        req = e.pool_req[j];
        pos = e.pool_pos[j];
      } else {
        req = j / e.rows_per_req;
        pos = e.pool_pos0[req] + j % e.rows_per_req;
      }
      if (pos < 0) {
        pg = -2;
      } else {
        const int pi = pos / e.page_size;
        pg = pi < e.max_pages ? e.page_table[static_cast<size_t>(req) * e.max_pages + pi] : -3;
        if (pg < 0 || pg >= e.n_pages) {
          raise_status(p.status, DFLASH_ERR_CAPACITY, 101);
          pg = -2;
        }
      }
    }
    r_req[r] = req;
    r_pos[r] = pos;
    r_pg[r] = pg;
  }
  float gq[4], gk[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int i = lane + 32 * t;
    gq[t] = (e.q_norm != nullptr && i < d) ? bf2f(e.q_norm[i]) : 1.f;
    gk[t] = (e.k_norm != nullptr && i < d) ? bf2f(e.k_norm[i]) : 1.f;
  }
  __syncthreads();
  for (int w = warp; w < rows * per_tile; w += 4) {
    const int r = w / per_tile, hl = w % per_tile;
    const int m = m0 + r;
    const int head = (e.f0 + tile * kTileN + hl * d) / d;
    const int kind = head < hq ? 0 : (head < hq + hkv ? 1 : 2);
    const int hidx = kind == 0 ? head : (kind == 1 ? head - hq : head - hq - hkv);
    const bool is_blk = m < e.n_blk;
    const int req = r_req[r], pos = r_pos[r], pg = r_pg[r];
    if (!is_blk) {
      if (pg == -2) continue;
      if (kind == 0 && !e.keep_q_pool) continue;
    }
    const float* xs = ts + r * C::TS_LD + hl * d;
    float x1[2], x2[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (t < npair) {
        x1[t] = xs[lane + 32 * t];
        x2[t] = xs[lane + 32 * t + half];
      }
    }
    if (kind < 2) {
      const bool norm = kind == 0 ? (e.q_norm != nullptr) : (e.k_norm != nullptr);
      if (norm) {
        float ss = 0.f;
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (t < npair) ss += x1[t] * x1[t] + x2[t] * x2[t];
        ss = warp_sum(ss);
        const float inv = rsqrtf(ss / static_cast<float>(d) + e.eps);
        // gain index lane+32t lives in slot t; its rotate-half partner in slot t + npair
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (t < npair) {
            const float ga = kind == 0 ? gq[t] : gk[t];
            const float gb = kind == 0 ? gq[t + npair] : gk[t + npair];
            x1[t] = x1[t] * inv * ga;
            x2[t] = x2[t] * inv * gb;
          }
        }
      }
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (t < npair) {
          float sn, cs;
          rope_sincos(pos, e.rope[lane + 32 * t], &sn, &cs);
          const float a = x1[t], b = x2[t];
          x1[t] = a * cs - b * sn;
          x2[t] = b * cs + a * sn;
        }
      }
    }
    uint16_t* dst;
    if (kind == 0) {
      dst = e.q + (static_cast<size_t>(m) * hq + hidx) * d;
    } else if (is_blk) {
      dst = (kind == 1 ? e.kblk : e.vblk) +
            ((static_cast<size_t>(req) * hkv + hidx) * e.block + m % e.block) * d;
    } else {
      dst = e.pool + ((((static_cast<size_t>(pg) * 2 + (kind - 1)) * hkv + hidx) * e.page_size) +
                      pos % e.page_size) * d;
    }
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (t < npair) {
        dst[lane + 32 * t] = f2bf(x1[t]);
        dst[lane + 32 * t + half] = f2bf(x2[t]);
      }
    }
  }
}

// ---------------------------------------------------------------- kernel
template <int BN>
__global__ void __launch_bounds__(128, 1)
    gemm_tc05_kernel(const __grid_constant__ CUtensorMap wmap,
                     const __grid_constant__ CUtensorMap xmap, const __grid_constant__ GemmParams p) {
  using C = GemmCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::MAIN_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* done = empty + C::STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);
  float* ts = reinterpret_cast<float*>(smem);  // staged tile (after the mainloop)

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int tile = blockIdx.x, split = blockIdx.y, mt = blockIdx.z;
  const int m0 = mt * BN;
  const int kb0 = split * p.kb_per_split;
  const int kb1 = min(p.kb_total, kb0 + p.kb_per_split);
  const int nkb = kb1 - kb0;

  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    *last_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&wmap);
    tma_prefetch_desc(&xmap);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  griddep_launch_dependents();

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_x = l2_policy_evict_last();
    const int wrow = p.w_row0 + tile * p.w_tile_step;
    const int pre = nkb < C::STAGES ? nkb : C::STAGES;
    for (int it = 0; it < pre; ++it) {
      uint8_t* a = smem + it * C::A_BYTES;
      const int kx = (kb0 + it) * kTileK;
      mbar_arrive_expect_tx(&full[it], C::STAGE_BYTES);
      tma_load_2d(a, &wmap, kx, wrow, &full[it], pol_w);
      tma_load_2d(a + C::A_BYTES / 2, &wmap, kx, wrow + p.w_half_gap, &full[it], pol_w);
    }
    griddep_wait();  // activations come from the previous kernel
    for (int it = 0; it < pre; ++it) {
      uint8_t* b = smem + C::STAGES * C::A_BYTES + it * C::B_BYTES;
      tma_load_2d(b, &xmap, (kb0 + it) * kTileK, m0, &full[it], pol_x);
    }
    for (int it = pre; it < nkb; ++it) {
      const int s = it % C::STAGES;
      const uint32_t ph = ((it / C::STAGES) & 1) ^ 1;
      if (!mbar_wait(&empty[s], ph, abort_flag)) {
        *abort_flag = 1;
        raise_status(p.status, DFLASH_ERR_TIMEOUT, 11);
        break;
      }
      uint8_t* a = smem + s * C::A_BYTES;
      uint8_t* b = smem + C::STAGES * C::A_BYTES + s * C::B_BYTES;
      const int kx = (kb0 + it) * kTileK;
      mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
      tma_load_2d(a, &wmap, kx, wrow, &full[s], pol_w);
      tma_load_2d(a + C::A_BYTES / 2, &wmap, kx, wrow + p.w_half_gap, &full[s], pol_w);
      tma_load_2d(b, &xmap, kx, m0, &full[s], pol_x);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer (single thread)
    constexpr uint32_t idesc = umma_idesc_bf16(kTileN, BN);
    for (int it = 0; it < nkb; ++it) {
      const int s = it % C::STAGES;
      const uint32_t ph = (it / C::STAGES) & 1;
      if (!mbar_wait(&full[s], ph, abort_flag)) {
        *abort_flag = 1;
        raise_status(p.status, DFLASH_ERR_TIMEOUT, 12);
        break;
      }
      tc_fence_after();
      const uint64_t ad = umma_desc_sw128(smem_u32(smem + s * C::A_BYTES));
      const uint64_t bd = umma_desc_sw128(smem_u32(smem + C::STAGES * C::A_BYTES + s * C::B_BYTES));
#pragma unroll
      for (int k = 0; k < kTileK / 16; ++k)
        umma_bf16(tmem, ad + 2 * k, bd + 2 * k, idesc, (it | k) != 0 ? 1u : 0u);
      umma_commit(&empty[s]);
    }
    umma_commit(done);
  }
  if (!(warp == 0 && lane == 0)) griddep_wait();
  __syncwarp();

  // ---------------- epilogue: TMEM -> (partials | staged tile)
  const bool ok = mbar_wait(done, 0, abort_flag);
  if (!ok) {
    *abort_flag = 1;
    if (lane == 0) raise_status(p.status, DFLASH_ERR_TIMEOUT, 13);
  }
  __syncthreads();
  const bool aborted = *abort_flag != 0;
  tc_fence_after();
  const int rows = min(BN, p.M - m0);
  const int f = warp * 32 + lane;
  const int n0 = tile * kTileN;
  bool do_epi = false;
  // rows of the tile this CTA finishes: all of them without split-K; with
  // split-K the S CTAs of the tile form one cluster and CTA q finishes rows
  // [q*rpc, q*rpc + rpc) (request-aligned when the block conv couples rows)
  int r_beg = 0, r_cnt = rows;
  if (p.splits == 1) {
    if (!aborted) {
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        float v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c * 16, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) ts[(c * 16 + j) * C::TS_LD + f] = v[j];
      }
      do_epi = true;
    }
  } else if (!p.cluster) {
    // Split-K through global memory: every CTA stores its fp32 partial tile;
    // the last CTA of the tile (atomic ticket, no waiting) sums the partials
    // in split order and finishes the whole tile.
    if (!aborted) {
      float* part = p.partial + static_cast<size_t>(split) * p.M * p.N;
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        float v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c * 16, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int r = c * 16 + j;
          if (r < rows) part[static_cast<size_t>(m0 + r) * p.N + n0 + f] = v[j];
        }
      }
      __threadfence();
    }
    __syncthreads();
    if (tid == 0) {
      const int prev = aborted ? 0 : atomicAdd(&p.counters[mt * gridDim.x + tile], 1);
      *last_flag = (!aborted && prev == p.splits - 1) ? 1 : 0;
    }
    __syncthreads();
    if (*last_flag) {
      __threadfence();
      const size_t sstride = static_cast<size_t>(p.M) * p.N / 4;  // float4 per split
      const float4* pbase = reinterpret_cast<const float4*>(p.partial);
      const int nchunk = rows * 32;
      for (int c0 = tid; c0 < nchunk; c0 += 4 * 128) {
        // up to 4 chunks per thread, splits in groups of 4: 16 loads in flight
        const float4* src[4];
        float4 acc[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = c0 + i * 128;
          src[i] = pbase + (static_cast<size_t>(m0 + (c < nchunk ? c / 32 : 0)) * p.N + n0) / 4 + c % 32;
          acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        int sp = 0;
        for (; sp + 4 <= p.splits; sp += 4) {
          float4 v[4][4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
              v[i][j] = (c0 + i * 128 < nchunk) ? __ldcg(src[i] + (sp + j) * sstride)
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              acc[i].x += v[i][j].x; acc[i].y += v[i][j].y;
              acc[i].z += v[i][j].z; acc[i].w += v[i][j].w;
            }
        }
        for (; sp < p.splits; ++sp) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (c0 + i * 128 < nchunk) {
              const float4 v = __ldcg(src[i] + sp * sstride);
              acc[i].x += v.x; acc[i].y += v.y; acc[i].z += v.z; acc[i].w += v.w;
            }
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = c0 + i * 128;
          if (c < nchunk)
            *reinterpret_cast<float4*>(ts + (c / 32) * C::TS_LD + (c % 32) * 4) = acc[i];
        }
      }
      if (tid == 0) p.counters[mt * gridDim.x + tile] = 0;
      __syncthreads();
      do_epi = true;
    }
  } else {
    // 1) own partial tile -> own shared memory
    if (!aborted) {
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        float v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c * 16, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) ts[(c * 16 + j) * C::TS_LD + f] = v[j];
      }
    }
    cluster_sync();
    // 2) reduce this CTA's rows over the cluster's partials (split order)
    const int S = p.splits;
    const int q = static_cast<int>(cluster_ctarank());
    int rpc = (rows + S - 1) / S;
    if (p.conv != nullptr && p.conv_width > 0) rpc = (rpc + p.block - 1) / p.block * p.block;
    r_beg = min(rows, q * rpc);
    r_cnt = min(rows, r_beg + rpc) - r_beg;
    // Peers read only rows of their own range from this CTA's tile and this
    // CTA overwrites only rows of its range, so the in-place write needs no
    // extra barrier; the final cluster barrier keeps every tile alive until
    // all peers are done reading.
    const uint32_t ts_addr = smem_u32(ts);
    const int nchunk = r_cnt * 32;  // float4 chunks of my rows
    for (int c0 = tid; c0 < nchunk; c0 += 4 * 128) {
      float4 red[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) red[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int sp = 0; sp < S; ++sp) {
        const uint32_t peer = dsmem_map(ts_addr, static_cast<uint32_t>(sp));
        float4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = c0 + i * 128;
          v[i] = c < nchunk
                     ? dsmem_ld4(peer + static_cast<uint32_t>(((r_beg + c / 32) * C::TS_LD + (c % 32) * 4) * 4))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          red[i].x += v[i].x; red[i].y += v[i].y; red[i].z += v[i].z; red[i].w += v[i].w;
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = c0 + i * 128;
        if (c < nchunk)
          *reinterpret_cast<float4*>(ts + (r_beg + c / 32) * C::TS_LD + (c % 32) * 4) = red[i];
      }
    }
    __syncthreads();
    do_epi = !aborted && r_cnt > 0;
  }
  float* tsv = ts + r_beg * C::TS_LD;   // first row this CTA finishes
  const int m0v = m0 + r_beg;
  const int rows_v = r_cnt;
  if (do_epi && p.ssq_in != nullptr) {
    // one warp per row: the lanes read the row's per-tile sums together and
    // combine them with a fixed butterfly (same order for any M)
    float* rinv = reinterpret_cast<float*>(smem + C::SCRATCH_OFF);
    for (int r = warp; r < rows_v; r += 4) {
      const float* q = p.ssq_in + static_cast<size_t>(m0v + r) * p.ssq_in_tiles;
      float ss = 0.f;
      for (int t = lane; t < p.ssq_in_tiles; t += 32) ss += q[t];
      ss = warp_sum(ss);
      if (lane == 0)
        rinv[r] = (m0v + r < p.norm_rows) ? rsqrtf(ss / static_cast<float>(p.norm_dim) + p.norm_eps) : 1.f;
    }
    __syncthreads();
    for (int idx = tid; idx < rows_v * kTileN; idx += 128) {
      const int r = idx / kTileN, f = idx % kTileN;
      tsv[r * C::TS_LD + f] *= rinv[r];
    }
    __syncthreads();
  }
  if (do_epi) {
    switch (p.mode) {
      case EPI_STORE_BF16:
      case EPI_STORE_F32: epi_store<BN>(p, tsv, tile, m0v, rows_v); break;
      case EPI_RESID: epi_resid<BN>(p, tsv, tile, m0v, rows_v); break;
      case EPI_SWIGLU: epi_swiglu<BN>(p, tsv, tile, m0v, rows_v); break;
      case EPI_ARGMAX: epi_argmax<BN>(p, tsv, tile, m0v, rows_v); break;
      case EPI_QKV:
        epi_qkv<BN>(p, tsv, tile, m0v, rows_v, reinterpret_cast<int*>(smem + C::SCRATCH_OFF + BN * 4));
        break;
      default: break;
    }
  }
  if (p.splits > 1 && p.cluster) cluster_sync();  // peers may still read this CTA's tile until here
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ---------------------------------------------------------------- host side
int gemm_bn_for(int M) {
  return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
}

int gemm_max_smem_bytes() {
  int m = GemmCfg<16>::SMEM_BYTES;
  m = m > GemmCfg<32>::SMEM_BYTES ? m : GemmCfg<32>::SMEM_BYTES;
  m = m > GemmCfg<64>::SMEM_BYTES ? m : GemmCfg<64>::SMEM_BYTES;
  m = m > GemmCfg<128>::SMEM_BYTES ? m : GemmCfg<128>::SMEM_BYTES;
  m = m > GemmCfg<256>::SMEM_BYTES ? m : GemmCfg<256>::SMEM_BYTES;
  return m;
}

// Dynamic shared memory size, and the largest shared-memory carveout so that
// several CTAs (of this and of the next kernel) can be resident per SM.
template <int BN>
static cudaError_t set_gemm_attrs() {
  cudaError_t e = cudaFuncSetAttribute(gemm_tc05_kernel<BN>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       GemmCfg<BN>::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemm_tc05_kernel<BN>,
                              cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared);
}

template <int BN>
static cudaError_t launch_bn(const CUtensorMap* w_map, const CUtensorMap* x_map,
                             const GemmParams& p, cudaStream_t s, bool pdl) {
  using C = GemmCfg<BN>;
  static thread_local int attr_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_device != dev) {
    cudaError_t e = set_gemm_attrs<BN>();
    if (e != cudaSuccess) return e;
    attr_device = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.N / kTileN, p.splits, (p.M + BN - 1) / BN);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[3];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (p.splits > 1 && p.cluster) {
    // the split-K CTAs of one output tile form a cluster (reduced through DSMEM)
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = p.splits;
    attr[na].val.clusterDim.z = 1;
    ++na;
    // let several CTAs of a cluster share an SM, so clusters of 8 do not cap
    // the number of resident CTAs
    attr[na].id = cudaLaunchAttributeClusterSchedulingPolicyPreference;
    attr[na].val.clusterSchedulingPolicyPreference = cudaClusterSchedulingPolicyLoadBalancing;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  count_launch();
  return cudaLaunchKernelEx(&cfg, gemm_tc05_kernel<BN>, *w_map, *x_map, p);
}

template <int BN>
static int max_clusters_bn(int cluster) {
  using C = GemmCfg<BN>;
  if (set_gemm_attrs<BN>() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, cluster, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = cluster;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_tc05_kernel<BN>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

int gemm_max_active_clusters(int bn, int cluster) {
  switch (bn) {
    case 16: return max_clusters_bn<16>(cluster);
    case 32: return max_clusters_bn<32>(cluster);
    case 64: return max_clusters_bn<64>(cluster);
    case 128: return max_clusters_bn<128>(cluster);
    case 256: return max_clusters_bn<256>(cluster);
    default: return 0;
  }
}

cudaError_t gemm_launch(const CUtensorMap* w_map, const CUtensorMap* x_map, const GemmParams& p,
                        int bn, cudaStream_t s, bool pdl) {
  switch (bn) {
    case 16: return launch_bn<16>(w_map, x_map, p, s, pdl);
    case 32: return launch_bn<32>(w_map, x_map, p, s, pdl);
    case 64: return launch_bn<64>(w_map, x_map, p, s, pdl);
    case 128: return launch_bn<128>(w_map, x_map, p, s, pdl);
    case 256: return launch_bn<256>(w_map, x_map, p, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dflash
