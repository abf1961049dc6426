// Attention building blocks of the mma.sync attention kernel (attention.cu).
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace dflash {


__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)),
               "l"(gsrc), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

constexpr int kChunk = 64;

// Physical page ids of one split's key range are staged in shared memory
// (one parallel round trip) instead of being looked up per 16-byte piece.
constexpr int kMaxSplitPages = 512;

// K/V chunk buffers of the cp.async pipeline (NBUF-1 chunks in flight ahead
// of the one being computed); TERMS = 2 adds the low-term buffers of K and V.
template <int D, int NBUF, int TERMS = 1>
__host__ __device__ constexpr int attn_kv_bytes() {
  return 2 /*K,V*/ * TERMS * NBUF * kChunk * D * 2;
}
template <int D, int NBUF, int TERMS = 1>
__host__ __device__ constexpr int attn_smem_bytes() {
  return attn_kv_bytes<D, NBUF, TERMS>() + kMaxSplitPages * 4;
}

// Byte offset of (key row, 16-byte column chunk) in a swizzled [64][D] tile.
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * (D * 2) + ((chunk ^ (row & 7)) << 4));
}

template <int D>
struct AttnAcc {
  float o[D / 8][4];
  float m[2], l[2];
  int row_lo, head;
};

// Attention of one work unit (request, KV head g, query tile qt, key split)
// over its key range, with NW warps (local thread index tid).  Leaves each
// warp's unnormalised O and running (m, l) of its 16 query rows in acc.
// Returns false when the query tile is past the request's rows.
// TERMS = 2: pool keys and values are hi + lo bf16 planes; S = Q K_hi^T +
// Q K_lo^T and O += P V_hi + P V_lo accumulate both terms in fp32 (the
// in-block keys of the drafter mode have one term: their lo tiles are zero).
template <int D, int NW, int NBUF, typename Sync, int TERMS = 1>
__device__ __forceinline__ bool attn_accumulate(const AttnParams& p, int split, int qt, int req,
                                                int g, int tid, uint8_t* sm, Sync sync,
                                                AttnAcc<D>& acc) {
  uint8_t* Kbuf = sm;
  uint8_t* Vbuf = sm + NBUF * kChunk * D * 2;
  uint8_t* Klo = sm + 2 * NBUF * kChunk * D * 2;  // TERMS = 2 only
  uint8_t* Vlo = sm + 3 * NBUF * kChunk * D * 2;

  const int G = p.hq / p.hkv;
  const int R = 16 * NW / G;  // query rows per CTA
  const int warp = tid / 32, lane = tid % 32;
  const int hl = warp % G, rg = warp / G;
  const int head = g * G + hl;
  const int row_lo = qt * R + rg * 16;  // first row (within the request) of this warp
  const int group = lane / 4, tq = lane % 4;

  if (qt * R >= p.n) return false;
  const int pos0 = p.pos0[req];
  const int S = p.split_keys;
  // key range of this split; an empty range leaves (m, l, O) = (-inf, 0, 0)
  int k_lo = 0, k_hi = 0;
  bool blk = false;
  if (p.causal) {
    const int last_row = min(p.n, (qt + 1) * R) - 1;
    const int kmax = pos0 + last_row + 1;
    if (split * S < kmax) {
      k_lo = split * S;
      k_hi = min(kmax, k_lo + S);
    }
  } else {
    const int nctx = (pos0 + S - 1) / S;
    if (split < nctx) {
      k_lo = split * S;
      k_hi = min(pos0, k_lo + S);
    } else if (split == nctx) {
      blk = true;
      k_lo = 0;
      k_hi = p.n;
    }
  }

  // ---- query fragments (A operand, row-major 16 x D per warp)
  uint32_t qf[D / 16][4];
  {
    const int r0 = row_lo + group, r1 = r0 + 8;
    const uint16_t* q0 = p.q + ((static_cast<size_t>(req) * p.n + r0) * p.hq + head) * D;
    const uint16_t* q1 = p.q + ((static_cast<size_t>(req) * p.n + r1) * p.hq + head) * D;
    const bool v0 = r0 < p.n, v1 = r1 < p.n;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int c = kk * 16 + tq * 2;
      // L2-coherent loads (q was written by the previous kernel)
      qf[kk][0] = v0 ? __ldcg(reinterpret_cast<const unsigned int*>(q0 + c)) : 0u;
      qf[kk][1] = v1 ? __ldcg(reinterpret_cast<const unsigned int*>(q1 + c)) : 0u;
      qf[kk][2] = v0 ? __ldcg(reinterpret_cast<const unsigned int*>(q0 + c + 8)) : 0u;
      qf[kk][3] = v1 ? __ldcg(reinterpret_cast<const unsigned int*>(q1 + c + 8)) : 0u;
    }
  }

  const size_t plane = static_cast<size_t>(p.hkv) * p.page_size * D;  // K->V plane distance
  // stage this split's page ids (context keys only)
  int* pages_s = reinterpret_cast<int*>(sm + attn_kv_bytes<D, NBUF, TERMS>());
  const int page_lo = k_lo / p.page_size;
  if (!blk && k_hi > k_lo) {
    const int npg = (k_hi - 1) / p.page_size + 1 - page_lo;  // <= kMaxSplitPages (host caps S)
    for (int i = tid; i < npg; i += NW * 32) {
      const int pi = page_lo + i;
      int pg = pi < p.max_pages ? p.page_table[static_cast<size_t>(req) * p.max_pages + pi] : -1;
      if (pg < 0 || pg >= p.n_pages) {
        raise_status(p.status, DFLASH_ERR_CAPACITY, 201);
        pg = -1;
      }
      pages_s[i] = pg;
    }
    sync();
  }
  auto load_chunk = [&](int buf, int kc) {
    constexpr int PIECES = kChunk * (D / 8);
    for (int pc = tid; pc < PIECES; pc += NW * 32) {
      const int kr = pc / (D / 8), ch = pc % (D / 8);
      const int key = kc + kr;
      const uint16_t* sk = p.q;  // any valid address for a zero-fill copy
      const uint16_t* sv = p.q;
      int bytes = 0, bytes_lo = 0;
      if (key < k_hi) {
        if (blk) {
          const size_t o = ((static_cast<size_t>(req) * p.hkv + g) * p.n + key) * D + ch * 8;
          sk = p.kblk + o;
          sv = p.vblk + o;
          bytes = 16;
        } else {
          const int pg = pages_s[key / p.page_size - page_lo];
          if (pg >= 0) {
            const size_t o = (static_cast<size_t>(pg) * 2 * TERMS * p.hkv + g) * p.page_size * D +
                             static_cast<size_t>(key % p.page_size) * D + ch * 8;
            sk = p.pool + o;
            sv = p.pool + o + plane;
            bytes = 16;
            bytes_lo = 16;
          }
        }
      }
      const uint32_t off = buf * kChunk * D * 2 + swz<D>(kr, ch);
      cp_async16(Kbuf + off, sk, bytes);
      cp_async16(Vbuf + off, sv, bytes);
      if constexpr (TERMS == 2) {
        cp_async16(Klo + off, bytes_lo ? sk + 2 * plane : p.q, bytes_lo);
        cp_async16(Vlo + off, bytes_lo ? sv + 2 * plane : p.q, bytes_lo);
      }
    }
    cp_async_commit();
  };

  const float sc = rsqrtf(static_cast<float>(D)) * 1.4426950408889634f;
  float (&o)[D / 8][4] = acc.o;
  float* m_r = acc.m;
  float* l_r = acc.l;
  m_r[0] = m_r[1] = -INFINITY;
  l_r[0] = l_r[1] = 0.f;
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  const int qpos0 = pos0 + row_lo + group;  // positions of this thread's two rows
  const int qpos1 = qpos0 + 8;
  const int nch = k_hi > k_lo ? (k_hi - k_lo + kChunk - 1) / kChunk : 0;
  // prologue: the first NBUF-1 chunks (empty groups keep the count uniform)
#pragma unroll
  for (int c = 0; c < NBUF - 1; ++c) {
    if (c < nch)
      load_chunk(c, k_lo + c * kChunk);
    else
      cp_async_commit();
  }
  for (int c = 0; c < nch; ++c) {
    // chunk c+NBUF-1 goes into the buffer freed at the end of iteration c-1
    if (c + NBUF - 1 < nch)
      load_chunk((c + NBUF - 1) % NBUF, k_lo + (c + NBUF - 1) * kChunk);
    else
      cp_async_commit();
    cp_async_wait<NBUF - 1>();
    sync();
    const int buf = c % NBUF;
    const int kc = k_lo + c * kChunk;
    const uint32_t kbase = smem_u32(Kbuf) + buf * kChunk * D * 2;
    const uint32_t vbase = smem_u32(Vbuf) + buf * kChunk * D * 2;

    // S = Q K^T for 64 keys: 8 n-tiles of 8 keys
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
    // k-steps outer, the 8 key tiles inner: consecutive MMAs write different
    // accumulators, so they issue back to back instead of waiting on each other
#pragma unroll
    for (int kk = 0; kk < D / 16; kk += 2) {
      uint32_t bb[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        ldsm_x4(kbase + swz<D>(j * 8 + (lane & 7), kk * 2 + (lane >> 3)), bb[j][0], bb[j][1],
                bb[j][2], bb[j][3]);
#pragma unroll
      for (int j = 0; j < 8; ++j) mma16816(s[j], qf[kk], bb[j][0], bb[j][1]);
#pragma unroll
      for (int j = 0; j < 8; ++j) mma16816(s[j], qf[kk + 1], bb[j][2], bb[j][3]);
      if constexpr (TERMS == 2) {
        const uint32_t klo = smem_u32(Klo) + buf * kChunk * D * 2;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          ldsm_x4(klo + swz<D>(j * 8 + (lane & 7), kk * 2 + (lane >> 3)), bb[j][0], bb[j][1],
                  bb[j][2], bb[j][3]);
#pragma unroll
        for (int j = 0; j < 8; ++j) mma16816(s[j], qf[kk], bb[j][0], bb[j][1]);
#pragma unroll
        for (int j = 0; j < 8; ++j) mma16816(s[j], qf[kk + 1], bb[j][2], bb[j][3]);
      }
    }
    // mask + scale (log2 domain)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int kidx = kc + j * 8 + tq * 2 + (e & 1);
        bool ok = kidx < k_hi;
        if (p.causal) ok = ok && kidx <= (e < 2 ? qpos0 : qpos1);
        s[j][e] = ok ? s[j][e] * sc : -INFINITY;
      }
    }
    // online softmax, rows (group) and (group + 8)
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fmaxf(s[j][2 * rr], s[j][2 * rr + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_r[rr], mx);
      const bool dead = (m_new == -INFINITY);
      const float alpha = dead ? 1.f : exp2f(m_r[rr] - m_new);
      float rs = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float p0 = dead ? 0.f : exp2f(s[j][2 * rr] - m_new);
        const float p1 = dead ? 0.f : exp2f(s[j][2 * rr + 1] - m_new);
        s[j][2 * rr] = p0;
        s[j][2 * rr + 1] = p1;
        rs += p0 + p1;
      }
      rs += __shfl_xor_sync(0xffffffffu, rs, 1);
      rs += __shfl_xor_sync(0xffffffffu, rs, 2);
      l_r[rr] = l_r[rr] * alpha + rs;
      m_r[rr] = m_new;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        o[i][2 * rr] *= alpha;
        o[i][2 * rr + 1] *= alpha;
      }
    }
    // O += P V: 4 k-steps of 16 keys
#pragma unroll
    for (int kk = 0; kk < kChunk / 16; ++kk) {
      uint32_t a[4];
      a[0] = pack_bf2(s[2 * kk][0], s[2 * kk][1]);
      a[1] = pack_bf2(s[2 * kk][2], s[2 * kk][3]);
      a[2] = pack_bf2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      a[3] = pack_bf2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int nd = 0; nd < D / 8; nd += 2) {
        uint32_t b0, b1, b2, b3;
        const int krow = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        ldsm_x4_t(vbase + swz<D>(krow, nd + (lane >> 4)), b0, b1, b2, b3);
        mma16816(o[nd], a, b0, b1);
        mma16816(o[nd + 1], a, b2, b3);
        if constexpr (TERMS == 2) {
          const uint32_t vlo = smem_u32(Vlo) + buf * kChunk * D * 2;
          ldsm_x4_t(vlo + swz<D>(krow, nd + (lane >> 4)), b0, b1, b2, b3);
          mma16816(o[nd], a, b0, b1);
          mma16816(o[nd + 1], a, b2, b3);
        }
      }
    }
    sync();
  }
  acc.row_lo = row_lo;
  acc.head = head;
  return true;
}

// Unnormalised O and (m, l) of one warp's 16 query rows -> global partials.
template <int D>
__device__ __forceinline__ void attn_store_partial(const AttnParams& p, int split, int req,
                                                   const AttnAcc<D>& acc, int lane) {
  const int group = lane / 4, tq = lane % 4;
  const int rows_total = p.batch * p.n;
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int row = acc.row_lo + group + rr * 8;
    if (row >= p.n) continue;
    const size_t vid = (static_cast<size_t>(split) * rows_total + static_cast<size_t>(req) * p.n + row) * p.hq + acc.head;
    float* op = p.o_part + vid * D;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      const int col = i * 8 + tq * 2;
      *reinterpret_cast<float2*>(op + col) = make_float2(acc.o[i][2 * rr], acc.o[i][2 * rr + 1]);
    }
    if (tq == 0) {
      p.ml_part[vid * 2 + 0] = acc.m[rr];
      p.ml_part[vid * 2 + 1] = acc.l[rr];
    }
  }
}

// Merge the key splits of one query vector (row, head) in split order and
// write the normalised bf16 output; one warp, lane = lane index.
template <int D>
__device__ __forceinline__ void attn_combine_vec(const AttnParams& p, int vec, int lane) {
  const int rows_total = p.batch * p.n;
  const int row = vec / p.hq, head = vec % p.hq;
  const int req = row / p.n, i = row % p.n;
  const int pos0 = p.pos0[req];
  const int S = p.split_keys;
  const int ns = p.causal ? (pos0 + i + 1 + S - 1) / S : (pos0 + S - 1) / S + 1;
  const size_t vstride = static_cast<size_t>(rows_total) * p.hq;  // vectors per split
  const size_t v0 = static_cast<size_t>(row) * p.hq + head;
  float mstar = -INFINITY;
  for (int s0 = 0; s0 < ns; s0 += 32) {
    const float ms = (s0 + lane < ns) ? __ldcg(p.ml_part + ((s0 + lane) * vstride + v0) * 2) : -INFINITY;
    mstar = fmaxf(mstar, warp_max(ms));
  }
  float acc[D / 32];
#pragma unroll
  for (int t = 0; t < D / 32; ++t) acc[t] = 0.f;
  float lsum = 0.f;
  for (int s0 = 0; s0 < ns; s0 += 32) {
    const int sl = s0 + lane;
    float ms = -INFINITY, ls = 0.f;
    if (sl < ns) {
      ms = __ldcg(p.ml_part + (sl * vstride + v0) * 2);
      ls = __ldcg(p.ml_part + (sl * vstride + v0) * 2 + 1);
    }
    const float w = (ms == -INFINITY) ? 0.f : exp2f(ms - mstar);
    const int cnt = min(32, ns - s0);
    for (int j0 = 0; j0 < cnt; j0 += 8) {
      float v[8][D / 32];
      float wj[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        wj[j] = __shfl_sync(0xffffffffu, w, (j0 + j) & 31);
        const bool ok = j0 + j < cnt;
#pragma unroll
        for (int t = 0; t < D / 32; ++t)
          v[j][t] = ok ? __ldcg(p.o_part + ((s0 + j0 + j) * vstride + v0) * D + lane + 32 * t) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j0 + j < cnt) {
#pragma unroll
          for (int t = 0; t < D / 32; ++t) acc[t] += v[j][t] * wj[j];
        }
      }
    }
    // l in split order (lane order)
    float lw = ls * w;
    for (int j = 0; j < cnt; ++j) lsum += __shfl_sync(0xffffffffu, lw, j);
  }
  const float inv = 1.f / lsum;
  const size_t ob = (static_cast<size_t>(row) * p.hq + head) * D;
#pragma unroll
  for (int t = 0; t < D / 32; ++t) {
    const float v = acc[t] * inv;
    const uint16_t hi = f2bf(v);
    p.out[ob + lane + 32 * t] = hi;
    if (p.out_lo != nullptr) p.out_lo[ob + lane + 32 * t] = bf16_lo_part(v, hi);
  }
}

}  // namespace dflash
