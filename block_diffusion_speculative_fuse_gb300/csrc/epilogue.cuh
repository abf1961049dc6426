// Fused GEMM epilogues, shared by the per-GEMM kernel (gemm_tc05.cu) and the
// persistent layer-stack kernel (persistent_stack.cu).  Each works on a staged
// fp32 tile ts[rows][kTsLd] (rows = activation rows, 128 output features) with
// 128 cooperating threads (local index tid, 0..127, warp-aligned) and a
// caller-supplied barrier over those threads.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace dflash {

constexpr int kTsLd = kTileN + 4;  // staged tile row stride (floats)

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
template <typename Sync>
__device__ void epi_store(const GemmParams& p, const float* ts, int tile, int m0, int rows,
                          int tid, Sync sync) {
    const int n0 = tile * kTileN;
  for (int idx = tid; idx < rows * kTileN; idx += 128) {
    const int r = idx / kTileN, f = idx % kTileN;
    const float v = ts[r * kTsLd + f];
    const size_t o = static_cast<size_t>(m0 + r) * p.ld_out + n0 + f;
    if (p.mode == EPI_STORE_BF16)
      static_cast<uint16_t*>(p.out)[o] = f2bf(v);
    else
      static_cast<float*>(p.out)[o] = v;
  }
}

template <typename Sync>
__device__ void epi_resid(const GemmParams& p, float* ts, int tile, int m0, int rows,
                          int tid, Sync sync) {
    // Thread f owns feature column n0 + f: x_new = x + acc, then the optional
  // depthwise conv along block positions (sliding window down the column,
  // zero padded at each request's block edges), then the next norm's inputs.
  const int f = tid;
  const int n = tile * kTileN + f;
  for (int r0 = 0; r0 < rows; r0 += 16) {
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      v[j] = (r0 + j < rows) ? __ldcg(p.resid + static_cast<size_t>(m0 + r0 + j) * p.ld_resid + n) : 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (r0 + j < rows) ts[(r0 + j) * kTsLd + f] += v[j];
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
        win[j] = (j < p.conv_width && src >= 0 && src < p.block) ? ts[(r0 + src) * kTsLd + f] : 0.f;
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
          const float v = (nxt < p.block) ? ts[(r0 + nxt) * kTsLd + f] : 0.f;
          // window length is conv_width; keep the slot after the last live one
          win[p.conv_width - 1] = v;
        }
        ts[(r0 + i) * kTsLd + f] = y;
      }
    }
  }
  for (int r = 0; r < rows; ++r) {
    const float x = ts[r * kTsLd + f];
    const size_t m = static_cast<size_t>(m0 + r);
    p.resid[m * p.ld_resid + n] = x;
    if (p.xg_out != nullptr) {
      const float xg = x * bf2f(p.gnext[n]);
      const uint16_t hi = f2bf(xg);
      p.xg_out[m * p.ld_xg + n] = hi;
      if (p.xg_lo != nullptr) p.xg_lo[m * p.ld_xg + n] = bf16_lo_part(xg, hi);
    }
    if (p.raw_out != nullptr) p.raw_out[m * p.ld_raw + n] = f2bf(x);
  }
  if (p.ssq_out != nullptr) {
    sync();
    const int warp = tid / 32, lane = tid % 32;
    for (int r = warp; r < rows; r += 4) {
      float ss = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float v = ts[r * kTsLd + lane + 32 * k];
        ss = fmaf(v, v, ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) p.ssq_out[static_cast<size_t>(m0 + r) * p.ssq_ld + tile] = ss;
    }
  }
}

template <typename Sync>
__device__ void epi_swiglu(const GemmParams& p, const float* ts, int tile, int m0, int rows,
                           int tid, Sync sync) {
    uint16_t* out = static_cast<uint16_t*>(p.out);
  for (int idx = tid; idx < rows * 64; idx += 128) {
    const int r = idx / 64, j = idx % 64;
    const float g = ts[r * kTsLd + j];
    const float u = ts[r * kTsLd + 64 + j];
    const float h = silu_f(g) * u;
    const size_t o = static_cast<size_t>(m0 + r) * p.ld_out + tile * 64 + j;
    const uint16_t hi = f2bf(h);
    out[o] = hi;
    if (p.out_lo != nullptr) p.out_lo[o] = bf16_lo_part(h, hi);
  }
}

template <typename Sync>
__device__ void epi_argmax(const GemmParams& p, const float* ts, int tile, int m0, int rows,
                           int tid, Sync sync, int n_tiles) {
    const int warp = tid / 32, lane = tid % 32;
  const int n0 = tile * kTileN;
  if (rows > 32) {
    // one thread per row, features in increasing order: the first maximum
    // is the lowest index, the same (value, index) as the warp reduction
    for (int r = tid; r < rows; r += 128) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      const float4* row = reinterpret_cast<const float4*>(ts + r * kTsLd);
#pragma unroll 8
      for (int c4 = 0; c4 < kTileN / 4; ++c4) {
        const float4 v = row[c4];
        if (v.x > bv) { bv = v.x; bi = n0 + 4 * c4; }
        if (v.y > bv) { bv = v.y; bi = n0 + 4 * c4 + 1; }
        if (v.z > bv) { bv = v.z; bi = n0 + 4 * c4 + 2; }
        if (v.w > bv) { bv = v.w; bi = n0 + 4 * c4 + 3; }
      }
      p.amax_val[static_cast<size_t>(m0 + r) * n_tiles + tile] = bv;
      p.amax_idx[static_cast<size_t>(m0 + r) * n_tiles + tile] = bi;
    }
  }
  for (int r = warp; r < (rows > 32 ? 0 : rows); r += 4) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int f = lane + 32 * t;
      const float v = ts[r * kTsLd + f];
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
    for (int idx = tid; idx < rows * kTileN; idx += 128) {
      const int r = idx / kTileN, f = idx % kTileN;
      p.logits[static_cast<size_t>(m0 + r) * p.ld_logits + n0 + f] = ts[r * kTsLd + f];
    }
  }
}

// route: int scratch of 3 * route_cap entries (route_cap >= rows)
template <typename Sync>
__device__ void epi_qkv(const GemmParams& p, const float* ts, int tile, int m0, int rows,
                        int* route, int route_cap, int tid, Sync sync) {
    const QkvEpi& e = p.qkv;
  const int warp = tid / 32, lane = tid % 32;
  const int d = e.head_dim;
  const int half = d / 2;
  const int per_tile = kTileN / d;
  const int npair = half / 32;  // pairs per lane: 1 (d=64) or 2 (d=128)
  const int hq = e.n_q_heads, hkv = e.n_kv_heads;
  // Per-row routing, one thread per row, all lookups issued in parallel:
  // route[r] = (request, position, physical page or -1 for block rows / -2 skip)
  int* r_req = route;
  int* r_pos = route + route_cap;
  int* r_pg = route + 2 * route_cap;
  for (int r = tid; r < rows; r += 128) {
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
  sync();
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
    const float* xs = ts + r * kTsLd + hl * d;
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

}  // namespace dflash
