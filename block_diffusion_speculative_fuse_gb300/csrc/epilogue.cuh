// Fused GEMM epilogues of the tcgen05 GEMM (gemm_tc05.cu).  Each works on a staged
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
// reduced angle is accurate to ~1e-6 rad for positions up to 2^24; its sine
// and cosine come from the hardware approximation, whose absolute error on
// [-pi, pi] (below 2^-21.4, per NVIDIA's documentation of __sincosf) is
// smaller than the angle's.
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
  __sincosf(r, s, c);
}

// ---------------------------------------------------------------- argmax keys
// (value, index) as one unsigned 64-bit key whose integer order is: larger
// value first, then lower index.  The value's bits are mapped to an unsigned
// integer of the same order (negative: all bits flipped; otherwise the sign
// bit set); -0 is taken as +0 so that the two zeros tie like in a float
// comparison.
__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
  if (v == 0.f) v = 0.f;
  const uint32_t b = __float_as_uint(v);
  const uint32_t o = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<unsigned long long>(o) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(idx));
}
__device__ __forceinline__ int argmax_key_index(unsigned long long k) {
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull));
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

// pre_resid (nullable): the residual rows m0 .. m0+rows-1 of this tile's 128
// columns, already loaded ([rows][128]); pre_g (nullable): gnext of the tile.
// x_new = x + acc, then the optional depthwise conv along block positions
// (sliding window down each column, zero padded at each request's block
// edges), then the outputs: x_new (fp32), the next norm's input
// bf16(x_new * gnext) (+ its low term), bf16(x_new) for taps, and the row's
// sum of squares over the tile.
template <typename Sync>
__device__ void epi_resid(const GemmParams& p, float* ts, int tile, int m0, int rows,
                          int tid, Sync sync, const float* pre_resid = nullptr,
                          const float* pre_g = nullptr) {
  const int warp = tid / 32, lane = tid % 32;
  const int n0 = tile * kTileN;
  const bool conv = p.conv != nullptr && p.conv_width > 0;
  bool added = false;  // residual already in ts
  if (pre_resid != nullptr) {
    for (int r = 0; r < rows; ++r) ts[r * kTsLd + tid] += pre_resid[r * kTileN + tid];
    added = true;
  } else if (conv) {
    // the conv needs whole columns: the tile's residual rows as 16-byte
    // pieces first, 16 loads in flight per thread, added where they land
    const float* rbase = p.resid + static_cast<size_t>(m0) * p.ld_resid + n0;
    const int pieces = rows * (kTileN / 4);
    for (int c0 = tid; c0 < pieces; c0 += 128 * 16) {
      float4 v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int c = c0 + i * 128;
        if (c < pieces)
          v[i] = __ldcg(reinterpret_cast<const float4*>(rbase + static_cast<size_t>(c / 32) * p.ld_resid) + c % 32);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int c = c0 + i * 128;
        if (c < pieces) {
          float4* t = reinterpret_cast<float4*>(ts + (c / 32) * kTsLd + (c % 32) * 4);
          float4 x = *t;
          x.x += v[i].x; x.y += v[i].y; x.z += v[i].z; x.w += v[i].w;
          *t = x;
        }
      }
    }
    added = true;
  }
  if (conv) {
    sync();
    // thread f slides the window down feature column n0 + f
    const int f = tid;
    const int n = n0 + f;
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
        const float v = (nxt < p.block) ? ts[(r0 + nxt) * kTsLd + f] : 0.f;
        win[p.conv_width - 1] = v;  // window length is conv_width
        ts[(r0 + i) * kTsLd + f] = y;
      }
    }
  }
  sync();  // every column complete before the row-wise output pass
  // Outputs: warp w takes rows w*4 .. w*4+3 of every 16, lane l columns
  // 4l .. 4l+3 (16-byte fp32 and 8-byte bf16 stores; the row's sum of
  // squares is the warp sum of the lanes' 4-term sums).
  float gn[4] = {0.f, 0.f, 0.f, 0.f};
  if (p.xg_out != nullptr) {
#pragma unroll
    for (int k = 0; k < 4; ++k) gn[k] = pre_g != nullptr ? pre_g[4 * lane + k] : bf2f(p.gnext[n0 + 4 * lane + k]);
  }
  for (int r0 = warp * 4; r0 < rows; r0 += 16) {
    float4 res[4];
    if (!added) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        res[i] = r0 + i < rows ? __ldcg(reinterpret_cast<const float4*>(
                                     p.resid + static_cast<size_t>(m0 + r0 + i) * p.ld_resid + n0) + lane)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = r0 + i;
      if (r >= rows) break;  // warp-uniform
      float4 x = *reinterpret_cast<const float4*>(ts + r * kTsLd + 4 * lane);
      if (!added) {
        x.x += res[i].x; x.y += res[i].y; x.z += res[i].z; x.w += res[i].w;
      }
      const size_t m = static_cast<size_t>(m0 + r);
      *reinterpret_cast<float4*>(p.resid + m * p.ld_resid + n0 + 4 * lane) = x;
      const float xv[4] = {x.x, x.y, x.z, x.w};
      if (p.xg_out != nullptr) {
        uint16_t hi[4], lo[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float xg = xv[k] * gn[k];
          hi[k] = f2bf(xg);
          lo[k] = bf16_lo_part(xg, hi[k]);
        }
        const size_t o = m * p.ld_xg + n0 + 4 * lane;
        *reinterpret_cast<uint2*>(p.xg_out + o) =
            make_uint2(hi[0] | (static_cast<uint32_t>(hi[1]) << 16), hi[2] | (static_cast<uint32_t>(hi[3]) << 16));
        if (p.xg_lo != nullptr)
          *reinterpret_cast<uint2*>(p.xg_lo + o) =
              make_uint2(lo[0] | (static_cast<uint32_t>(lo[1]) << 16), lo[2] | (static_cast<uint32_t>(lo[3]) << 16));
      }
      if (p.raw_out != nullptr) {
        const size_t o = m * p.ld_raw + n0 + 4 * lane;
        *reinterpret_cast<uint2*>(p.raw_out + o) =
            make_uint2(f2bf(xv[0]) | (static_cast<uint32_t>(f2bf(xv[1])) << 16),
                       f2bf(xv[2]) | (static_cast<uint32_t>(f2bf(xv[3])) << 16));
      }
      if (p.ssq_out != nullptr) {
        float ss = xv[0] * xv[0];
        ss = fmaf(xv[1], xv[1], ss);
        ss = fmaf(xv[2], xv[2], ss);
        ss = fmaf(xv[3], xv[3], ss);
        ss = warp_sum(ss);
        if (lane == 0) p.ssq_out[m * p.ssq_ld + tile] = ss;
      }
    }
  }
}

template <typename Sync>
__device__ void epi_swiglu(const GemmParams& p, const float* ts, int tile, int m0, int rows,
                           int tid, Sync sync) {
  // Thread (row r, group q of 8) forms h = silu(g) * u for pairs 4q..4q+3
  // and 32+4q..32+4q+3 of the tile's 64: the 8 threads of a row read 128
  // contiguous bytes per 16-byte load and store 4 bf16 at a time.
  uint16_t* out = static_cast<uint16_t*>(p.out);
  for (int idx = tid; idx < rows * 8; idx += 128) {
    const int r = idx / 8, q = idx % 8;
    const float* tr = ts + r * kTsLd;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int j = half * 32 + q * 4;
      const float4 g = *reinterpret_cast<const float4*>(tr + j);
      const float4 u = *reinterpret_cast<const float4*>(tr + 64 + j);
      const float h[4] = {silu_f(g.x) * u.x, silu_f(g.y) * u.y, silu_f(g.z) * u.z, silu_f(g.w) * u.w};
      uint16_t hi[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) hi[k] = f2bf(h[k]);
      const size_t o = static_cast<size_t>(m0 + r) * p.ld_out + tile * 64 + j;
      *reinterpret_cast<uint2*>(out + o) =
          make_uint2(hi[0] | (static_cast<uint32_t>(hi[1]) << 16), hi[2] | (static_cast<uint32_t>(hi[3]) << 16));
      if (p.out_lo != nullptr) {
        uint16_t lo[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) lo[k] = bf16_lo_part(h[k], hi[k]);
        *reinterpret_cast<uint2*>(p.out_lo + o) =
            make_uint2(lo[0] | (static_cast<uint32_t>(lo[1]) << 16), lo[2] | (static_cast<uint32_t>(lo[3]) << 16));
      }
    }
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
      if (p.amax_key != nullptr) {
        atomicMax(p.amax_key + m0 + r, argmax_key(bv, bi));
      } else {
        p.amax_val[static_cast<size_t>(m0 + r) * n_tiles + tile] = bv;
        p.amax_idx[static_cast<size_t>(m0 + r) * n_tiles + tile] = bi;
      }
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
      if (p.amax_key != nullptr) {
        atomicMax(p.amax_key + m0 + r, argmax_key(bv, bi));
      } else {
        p.amax_val[static_cast<size_t>(m0 + r) * n_tiles + tile] = bv;
        p.amax_idx[static_cast<size_t>(m0 + r) * n_tiles + tile] = bi;
      }
    }
  }
  if (p.logits != nullptr) {
    for (int idx = tid; idx < rows * kTileN; idx += 128) {
      const int r = idx / kTileN, f = idx % kTileN;
      p.logits[static_cast<size_t>(m0 + r) * p.ld_logits + n0 + f] = ts[r * kTsLd + f];
    }
  }
}

// Routing of activation row m of the QKV epilogue: (request, position,
// physical page), page -1 for block rows, -2 for a skipped or invalid
// context row (an invalid request index or page id also raises
// DFLASH_ERR_CAPACITY).
__device__ __forceinline__ void qkv_route(const GemmParams& p, int m, int* req_out, int* pos_out,
                                          int* pg_out) {
  const QkvEpi& e = p.qkv;
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
    if (req < 0 || req >= e.n_req) {
      if (pos >= 0) raise_status(p.status, DFLASH_ERR_CAPACITY, 102);
      req = 0;
      pg = -2;
    } else if (pos < 0) {
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
  *req_out = req;
  *pos_out = pos;
  *pg_out = pg;
}

// route: int scratch of 3 * route_cap entries (route_cap >= rows); pre_route
// (nullable): the routing of rows m0.. already computed, with stride pre_cap;
// pre_gain / pre_cs (nullable): the tile's q/k-norm gains [d] and the RoPE
// (cos, sin) of rows m0.. [rows][64] already computed.
template <typename Sync>
__device__ void epi_qkv(const GemmParams& p, const float* ts, int tile, int m0, int rows,
                        int* route, int route_cap, int tid, Sync sync,
                        const int* pre_route = nullptr, int pre_cap = 0,
                        const float* pre_gain = nullptr, const float2* pre_cs = nullptr) {
    const QkvEpi& e = p.qkv;
  const int warp = tid / 32, lane = tid % 32;
  const int d = e.head_dim;
  const int half = d / 2;
  const int per_tile = kTileN / d;
  const int hq = e.n_q_heads, hkv = e.n_kv_heads;
  // Per-row routing, one thread per row, all lookups issued in parallel:
  // route[r] = (request, position, physical page or -1 for block rows / -2 skip)
  const int* r_req = route;
  const int* r_pos = route + route_cap;
  const int* r_pg = route + 2 * route_cap;
  if (pre_route != nullptr) {
    r_req = pre_route;
    r_pos = pre_route + pre_cap;
    r_pg = pre_route + 2 * pre_cap;
  } else {
    for (int r = tid; r < rows; r += 128)
      qkv_route(p, m0 + r, route + r, route + route_cap + r, route + 2 * route_cap + r);
  }
  // Each (row, head) item is handled by a group of 8 lanes, 4 items per warp
  // at a time: lane `sub` of the group owns the rotate-half pairs
  // [sub*P, sub*P + P), P = d/16, so its loads and stores are contiguous
  // vectors and the head's sum of squares takes a 3-step butterfly.
  const int grp = lane / 8, sub = lane % 8;
  const int P = half / 8;  // 4 (d = 64) or 8 (d = 128)
  const int c0 = sub * P;
  float gq1[8], gq2[8], gk1[8], gk2[8];
  float2 rf[8];
  if (pre_gain == nullptr) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const bool in = j < P;
      gq1[j] = (in && e.q_norm != nullptr) ? bf2f(e.q_norm[c0 + j]) : 1.f;
      gq2[j] = (in && e.q_norm != nullptr) ? bf2f(e.q_norm[half + c0 + j]) : 1.f;
      gk1[j] = (in && e.k_norm != nullptr) ? bf2f(e.k_norm[c0 + j]) : 1.f;
      gk2[j] = (in && e.k_norm != nullptr) ? bf2f(e.k_norm[half + c0 + j]) : 1.f;
      rf[j] = in ? e.rope[c0 + j] : make_float2(0.f, 0.f);
    }
  }
  sync();
  const int items = rows * per_tile;
  // The loop bound depends on the warp only, so every lane reaches the
  // shuffles; items past the end or skipped rows only drop their stores.
  // The next iteration's tile values and routing are read before this
  // iteration's global stores (loads are not moved across those stores), so
  // their latency overlaps this iteration's arithmetic.
  float nx1[8], nx2[8];
  int nreq = 0, npos = 0, npg = 0;
  auto fetch = [&](int w0n) {
    const int wn = w0n + grp;
    const bool in = wn < items;
    const int rn = in ? wn / per_tile : 0, hln = in ? wn % per_tile : 0;
    nreq = r_req[rn];
    npos = r_pos[rn];
    npg = r_pg[rn];
    const float* xs = ts + rn * kTsLd + hln * d + c0;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
      if (4 * q < P) {
        a = *reinterpret_cast<const float4*>(xs + 4 * q);
        b = *reinterpret_cast<const float4*>(xs + half + 4 * q);
      }
      nx1[4 * q] = a.x; nx1[4 * q + 1] = a.y; nx1[4 * q + 2] = a.z; nx1[4 * q + 3] = a.w;
      nx2[4 * q] = b.x; nx2[4 * q + 1] = b.y; nx2[4 * q + 2] = b.z; nx2[4 * q + 3] = b.w;
    }
  };
  if (warp * 4 < items) fetch(warp * 4);
  for (int w0 = warp * 4; w0 < items; w0 += 16) {
    const int w = w0 + grp;
    bool act = w < items;
    const int r = act ? w / per_tile : 0, hl = act ? w % per_tile : 0;
    const int m = m0 + r;
    const int head = (e.f0 + tile * kTileN + hl * d) / d;
    const int kind = head < hq ? 0 : (head < hq + hkv ? 1 : 2);
    const int hidx = kind == 0 ? head : (kind == 1 ? head - hq : head - hq - hkv);
    const bool is_blk = m < e.n_blk;
    const int req = nreq, pos = npos, pg = npg;
    float x1[8], x2[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      x1[j] = nx1[j];
      x2[j] = nx2[j];
    }
    if (w0 + 16 < items) fetch(w0 + 16);
    if (!is_blk && (pg == -2 || (kind == 0 && !e.keep_q_pool))) act = false;
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) ss += x1[j] * x1[j] + x2[j] * x2[j];  // zero past P
    ss += __shfl_xor_sync(0xffffffffu, ss, 4);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    if (kind < 2) {
      const bool norm = kind == 0 ? (e.q_norm != nullptr) : (e.k_norm != nullptr);
      const float inv = norm ? rsqrtf(ss / static_cast<float>(d) + e.eps) : 1.f;
      if (pre_gain != nullptr) {
        // gains of this head kind and (cos, sin) of this row, precomputed
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j < P) {
            const float a = x1[j] * inv * pre_gain[c0 + j];
            const float b = x2[j] * inv * pre_gain[half + c0 + j];
            const float2 t = pre_cs[r * 64 + c0 + j];
            x1[j] = a * t.x - b * t.y;
            x2[j] = b * t.x + a * t.y;
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j < P) {
            const float a = x1[j] * inv * (kind == 0 ? gq1[j] : gk1[j]);
            const float b = x2[j] * inv * (kind == 0 ? gq2[j] : gk2[j]);
            float sn, cs;
            rope_sincos(pos, rf[j], &sn, &cs);
            x1[j] = a * cs - b * sn;
            x2[j] = b * cs + a * sn;
          }
        }
      }
    }
    // E4M3 context cache: amax of the head vector's bf16 values over its 8
    // lanes (every lane takes part in the shuffles)
    float am = 0.f;
    if (e.pool8 != nullptr) {  // uniform over the kernel
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < P) am = fmaxf(am, fmaxf(fabsf(bf2f(f2bf(x1[j]))), fabsf(bf2f(f2bf(x2[j])))));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 4));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
    }
    if (!act) continue;
    if (kind > 0 && !is_blk && e.pool8 != nullptr) {
      const float scale = am > 0.f ? am / 448.f : 1.f;
      const size_t vecid = (static_cast<size_t>(pg) * 2 + (kind - 1)) * hkv * e.page_size +
                           static_cast<size_t>(hidx) * e.page_size + pos % e.page_size;
      uint8_t* d8 = e.pool8 + vecid * d + c0;
      uint16_t c1[4], c2[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        c1[j] = e4m3x2_encode(bf2f(f2bf(x1[2 * j])) / scale, bf2f(f2bf(x1[2 * j + 1])) / scale);
        c2[j] = e4m3x2_encode(bf2f(f2bf(x2[2 * j])) / scale, bf2f(f2bf(x2[2 * j + 1])) / scale);
      }
      if (P == 8) {
        *reinterpret_cast<uint2*>(d8) = make_uint2(c1[0] | (static_cast<uint32_t>(c1[1]) << 16),
                                                   c1[2] | (static_cast<uint32_t>(c1[3]) << 16));
        *reinterpret_cast<uint2*>(d8 + half) = make_uint2(c2[0] | (static_cast<uint32_t>(c2[1]) << 16),
                                                          c2[2] | (static_cast<uint32_t>(c2[3]) << 16));
      } else {
        *reinterpret_cast<uint32_t*>(d8) = c1[0] | (static_cast<uint32_t>(c1[1]) << 16);
        *reinterpret_cast<uint32_t*>(d8 + half) = c2[0] | (static_cast<uint32_t>(c2[1]) << 16);
      }
      if (sub == 0) e.scales8[vecid] = scale;
      continue;
    }
    uint16_t* dst;
    uint16_t* dst_lo = nullptr;  // low terms (two-term cache)
    if (kind == 0) {
      dst = e.q + (static_cast<size_t>(m) * hq + hidx) * d;
    } else if (is_blk) {
      dst = (kind == 1 ? e.kblk : e.vblk) +
            ((static_cast<size_t>(req) * hkv + hidx) * e.block + m % e.block) * d;
    } else {
      const int planes = 2 * e.kv_terms;
      const size_t plane = static_cast<size_t>(hkv) * e.page_size * d;
      dst = e.pool + ((((static_cast<size_t>(pg) * planes + (kind - 1)) * hkv + hidx) * e.page_size) +
                      pos % e.page_size) * d;
      if (e.kv_terms == 2) dst_lo = dst + 2 * plane + c0;
    }
    dst += c0;
    uint32_t u1[4], u2[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      u1[j] = pack_bf2(x1[2 * j], x1[2 * j + 1]);
      u2[j] = pack_bf2(x2[2 * j], x2[2 * j + 1]);
    }
    if (P == 8) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(u1[0], u1[1], u1[2], u1[3]);
      *reinterpret_cast<uint4*>(dst + half) = make_uint4(u2[0], u2[1], u2[2], u2[3]);
    } else {
      *reinterpret_cast<uint2*>(dst) = make_uint2(u1[0], u1[1]);
      *reinterpret_cast<uint2*>(dst + half) = make_uint2(u2[0], u2[1]);
    }
    if (dst_lo != nullptr) {
      // v = hi + lo with lo = bf16(v - hi)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        u1[j] = pack_bf2(x1[2 * j] - bf2f(static_cast<uint16_t>(u1[j] & 0xFFFFu)),
                         x1[2 * j + 1] - bf2f(static_cast<uint16_t>(u1[j] >> 16)));
        u2[j] = pack_bf2(x2[2 * j] - bf2f(static_cast<uint16_t>(u2[j] & 0xFFFFu)),
                         x2[2 * j + 1] - bf2f(static_cast<uint16_t>(u2[j] >> 16)));
      }
      if (P == 8) {
        *reinterpret_cast<uint4*>(dst_lo) = make_uint4(u1[0], u1[1], u1[2], u1[3]);
        *reinterpret_cast<uint4*>(dst_lo + half) = make_uint4(u2[0], u2[1], u2[2], u2[3]);
      } else {
        *reinterpret_cast<uint2*>(dst_lo) = make_uint2(u1[0], u1[1]);
        *reinterpret_cast<uint2*>(dst_lo + half) = make_uint2(u2[0], u2[1]);
      }
    }
  }
}

}  // namespace dflash
