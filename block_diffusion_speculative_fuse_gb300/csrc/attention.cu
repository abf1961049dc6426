// Split-KV grouped-query attention over a paged KV cache (+ in-block keys).
//
// One CTA = (request, KV head, query-row tile, key split).  Its warps hold the
// 16-row query fragments of the G = hq/hkv query heads that share the KV head,
// so every K/V byte staged in shared memory feeds G*rows query vectors.  Keys
// are streamed in 64-key chunks (four 16-position pages) with cp.async double
// buffering into XOR-swizzled shared memory; QK^T and PV run on mma.sync
// m16n8k16 (bf16 in, fp32 accumulate) and the softmax is the online
// (running max / running sum) form with quad warp-shuffle row reductions in
// the exp2 domain.
//
// Split boundaries are fixed absolute key positions, chunk boundaries are
// 64-aligned inside them and masked keys contribute exact zeros, so a query
// row's result does not depend on which other rows share its CTA (the target
// forward relies on this for bit-identical block verify vs token-by-token
// decode).  attn_combine merges the per-split (O, m, l) in split order.
//
// Modes
//   non-causal (drafter): block row i of request r sits at pos0[r] + i and
//     attends to context keys [0, pos0[r]) of the pool and to all n block keys
//     (split index ceil(pos0/S) holds the block keys).
//   causal (target):      row i at pos0[r] + i attends to pool keys
//     [0, pos0[r] + i] (its own K/V were written by the QKV epilogue).
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

template <int D>
__host__ __device__ constexpr int attn_smem_bytes() {
  return 2 /*K,V*/ * 2 /*buffers*/ * kChunk * D * 2;
}

// Byte offset of (key row, 16-byte column chunk) in a swizzled [64][D] tile.
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * (D * 2) + ((chunk ^ (row & 7)) << 4));
}

template <int D, int NW>
__global__ void __launch_bounds__(NW * 32) attn_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(128) uint8_t sm[];
  uint8_t* Kbuf = sm;
  uint8_t* Vbuf = sm + 2 * kChunk * D * 2;

  const int G = p.hq / p.hkv;
  const int R = 16 * NW / G;  // query rows per CTA
  const int split = blockIdx.x, qt = blockIdx.y;
  const int req = blockIdx.z / p.hkv, g = blockIdx.z % p.hkv;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int hl = warp % G, rg = warp / G;
  const int head = g * G + hl;
  const int row_lo = qt * R + rg * 16;  // first row (within the request) of this warp
  const int group = lane / 4, tq = lane % 4;

  griddep_launch_dependents();
  griddep_wait();
  if (qt * R >= p.n) return;  // uniform over the cluster (clusters span splits only)
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
  if (!p.cluster && k_hi <= k_lo) return;

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
      qf[kk][0] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + c) : 0u;
      qf[kk][1] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + c) : 0u;
      qf[kk][2] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + c + 8) : 0u;
      qf[kk][3] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + c + 8) : 0u;
    }
  }

  const size_t plane = static_cast<size_t>(p.hkv) * p.page_size * D;  // K->V plane distance
  auto load_chunk = [&](int buf, int kc) {
    constexpr int PIECES = kChunk * (D / 8);
    for (int pc = tid; pc < PIECES; pc += NW * 32) {
      const int kr = pc / (D / 8), ch = pc % (D / 8);
      const int key = kc + kr;
      const uint16_t* sk = p.q;  // any valid address for a zero-fill copy
      const uint16_t* sv = p.q;
      int bytes = 0;
      if (key < k_hi) {
        if (blk) {
          const size_t o = ((static_cast<size_t>(req) * p.hkv + g) * p.n + key) * D + ch * 8;
          sk = p.kblk + o;
          sv = p.vblk + o;
          bytes = 16;
        } else {
          const int pi = key / p.page_size;
          const int pg =
              pi < p.max_pages ? p.page_table[static_cast<size_t>(req) * p.max_pages + pi] : -1;
          if (pg >= 0 && pg < p.n_pages) {
            const size_t o = (static_cast<size_t>(pg) * 2 * p.hkv + g) * p.page_size * D +
                             static_cast<size_t>(key % p.page_size) * D + ch * 8;
            sk = p.pool + o;
            sv = p.pool + o + plane;
            bytes = 16;
          } else if (ch == 0) {
            raise_status(p.status, DFLASH_ERR_CAPACITY, 201);
          }
        }
      }
      const uint32_t off = buf * kChunk * D * 2 + swz<D>(kr, ch);
      cp_async16(Kbuf + off, sk, bytes);
      cp_async16(Vbuf + off, sv, bytes);
    }
    cp_async_commit();
  };

  const float sc = rsqrtf(static_cast<float>(D)) * 1.4426950408889634f;
  float m_r[2] = {-INFINITY, -INFINITY};
  float l_r[2] = {0.f, 0.f};
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  const int qpos0 = pos0 + row_lo + group;  // positions of this thread's two rows
  const int qpos1 = qpos0 + 8;
  const int nch = k_hi > k_lo ? (k_hi - k_lo + kChunk - 1) / kChunk : 0;
  if (nch > 0) load_chunk(0, k_lo);
  for (int c = 0; c < nch; ++c) {
    if (c + 1 < nch) {
      load_chunk((c + 1) & 1, k_lo + (c + 1) * kChunk);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const int buf = c & 1;
    const int kc = k_lo + c * kChunk;
    const uint32_t kbase = smem_u32(Kbuf) + buf * kChunk * D * 2;
    const uint32_t vbase = smem_u32(Vbuf) + buf * kChunk * D * 2;

    // S = Q K^T for 64 keys: 8 n-tiles of 8 keys
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int kk = 0; kk < D / 16; kk += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + swz<D>(j * 8 + (lane & 7), kk * 2 + (lane >> 3)), b0, b1, b2, b3);
        mma16816(s[j], qf[kk], b0, b1);
        mma16816(s[j], qf[kk + 1], b2, b3);
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
      }
    }
    __syncthreads();
  }

  if (p.cluster) {
    // ---- combine across the cluster (the key splits of this query tile):
    // stage unnormalised O and (m, l) in shared memory, then CTA q merges a
    // share of the tile's query vectors from every peer, in split order.
    constexpr int NV = 16 * NW;  // query vectors of the tile: (warp, row in 16)
    float* Os = reinterpret_cast<float*>(sm);
    float* MLs = Os + NV * D;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int lv = warp * 16 + group + rr * 8;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        const int col = i * 8 + tq * 2;
        *reinterpret_cast<float2*>(Os + lv * D + col) = make_float2(o[i][2 * rr], o[i][2 * rr + 1]);
      }
      if (tq == 0) {
        MLs[lv * 2 + 0] = m_r[rr];
        MLs[lv * 2 + 1] = l_r[rr];
      }
    }
    const int SC = gridDim.x;
    if (SC > 1) cluster_sync();
    else __syncthreads();
    const int q = SC > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int vpc = (NV + SC - 1) / SC;
    const uint32_t os_addr = smem_u32(Os), ml_addr = smem_u32(MLs);
    for (int lv = q * vpc + warp; lv < min(NV, (q + 1) * vpc); lv += NW) {
      const int w = lv / 16, r = lv % 16;
      const int row = qt * R + (w / G) * 16 + r;
      const int hd = g * G + (w % G);
      // lane s < SC fetches split s's (m, l)
      float ms = -INFINITY, ls = 0.f;
      if (lane < SC) {
        const uint32_t a = (SC > 1 ? dsmem_map(ml_addr, lane) : ml_addr) + lv * 8;
        float2 v;
        asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a) : "memory");
        ms = v.x;
        ls = v.y;
      }
      const float mstar = warp_max(ms);
      float acc[D / 32];
#pragma unroll
      for (int t = 0; t < D / 32; ++t) acc[t] = 0.f;
      float lsum = 0.f;
      for (int sp = 0; sp < SC; ++sp) {
        const float msp = __shfl_sync(0xffffffffu, ms, sp);
        const float lsp = __shfl_sync(0xffffffffu, ls, sp);
        if (msp == -INFINITY) continue;
        const float wgt = exp2f(msp - mstar);
        lsum += lsp * wgt;
        const uint32_t base = (SC > 1 ? dsmem_map(os_addr, sp) : os_addr) + (lv * D) * 4;
#pragma unroll
        for (int t = 0; t < D / 32; ++t) {
          float v;
          asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(base + (lane + 32 * t) * 4) : "memory");
          acc[t] += v * wgt;
        }
      }
      if (row < p.n) {
        const float inv = 1.f / lsum;
        uint16_t* out = p.out + ((static_cast<size_t>(req) * p.n + row) * p.hq + hd) * D;
#pragma unroll
        for (int t = 0; t < D / 32; ++t) out[lane + 32 * t] = f2bf(acc[t] * inv);
      }
    }
    if (SC > 1) cluster_sync();  // peers may still read this CTA's partials until here
    return;
  }

  // ---- partial results: unnormalised O, running max (log2 domain) and sum
  const int rows_total = p.batch * p.n;
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int row = row_lo + group + rr * 8;
    if (row >= p.n) continue;
    const size_t vid = (static_cast<size_t>(split) * rows_total + static_cast<size_t>(req) * p.n + row) * p.hq + head;
    float* op = p.o_part + vid * D;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      const int col = i * 8 + tq * 2;
      *reinterpret_cast<float2*>(op + col) = make_float2(o[i][2 * rr], o[i][2 * rr + 1]);
    }
    if (tq == 0) {
      p.ml_part[vid * 2 + 0] = m_r[rr];
      p.ml_part[vid * 2 + 1] = l_r[rr];
    }
  }
}

// One warp per (row, head): merge the splits that cover the row, in order.
// Lane s holds split s's (m, l) (splits in groups of 32); the O partials of a
// group are loaded together before they are accumulated in split order.
template <int D>
__global__ void __launch_bounds__(128) attn_combine_kernel(const __grid_constant__ AttnParams p) {
  griddep_launch_dependents();
  griddep_wait();
  const int rows_total = p.batch * p.n;
  const int vec = blockIdx.x * 4 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (vec >= rows_total * p.hq) return;
  const int row = vec / p.hq, head = vec % p.hq;
  const int req = row / p.n, i = row % p.n;
  const int pos0 = p.pos0[req];
  const int S = p.split_keys;
  const int ns = p.causal ? (pos0 + i + 1 + S - 1) / S : (pos0 + S - 1) / S + 1;
  const size_t vstride = static_cast<size_t>(rows_total) * p.hq;  // vectors per split
  const size_t v0 = static_cast<size_t>(row) * p.hq + head;
  float mstar = -INFINITY;
  for (int s0 = 0; s0 < ns; s0 += 32) {
    const float ms = (s0 + lane < ns) ? p.ml_part[((s0 + lane) * vstride + v0) * 2] : -INFINITY;
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
      ms = p.ml_part[(sl * vstride + v0) * 2];
      ls = p.ml_part[(sl * vstride + v0) * 2 + 1];
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
  uint16_t* out = p.out + (static_cast<size_t>(row) * p.hq + head) * D;
#pragma unroll
  for (int t = 0; t < D / 32; ++t) out[lane + 32 * t] = f2bf(acc[t] * inv);
}

size_t attention_part_floats(int n_splits, int rows, int hq, int d) {
  return static_cast<size_t>(n_splits) * rows * hq * (d + 2);
}

template <int D, int NW>
static cudaError_t launch_attn(const AttnParams& p, cudaStream_t s, bool pdl) {
  static thread_local int attr_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<D, NW>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         attn_smem_bytes<D>());
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_kernel<D, NW>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_kernel<D, NW>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    attr_device = dev;
  }
  const int G = p.hq / p.hkv;
  const int R = 16 * NW / G;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  if (pdl) attrs[na++] = attr[0];
  if (p.cluster && p.n_splits > 1) {
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = p.n_splits;
    attrs[na].val.clusterDim.y = 1;
    attrs[na].val.clusterDim.z = 1;
    ++na;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_splits, (p.n + R - 1) / R, p.batch * p.hkv);
  cfg.blockDim = dim3(NW * 32, 1, 1);
  cfg.dynamicSmemBytes = attn_smem_bytes<D>();
  cfg.stream = s;
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  count_launch();
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_kernel<D, NW>, p);
  if (e != cudaSuccess || p.cluster) return e;
  cudaLaunchConfig_t c2 = {};
  const int vecs = p.batch * p.n * p.hq;
  c2.gridDim = dim3((vecs + 3) / 4, 1, 1);
  c2.blockDim = dim3(128, 1, 1);
  c2.stream = s;
  c2.attrs = attr;
  c2.numAttrs = pdl ? 1 : 0;
  count_launch();
  return cudaLaunchKernelEx(&c2, attn_combine_kernel<D>, p);
}

bool attention_cluster_ok(int d, int hq, int hkv, int n_splits) {
  // clusters of up to 16 CTAs (non-portable size, supported on sm_103)
  // partials of a 4-warp tile (64 vectors x d fp32) are staged in the K/V
  // buffers; 8-warp tiles and more than 8 splits use the global combine
  return n_splits <= kMaxAttnCluster && (hq / hkv) <= 4 && (d == 64 || d == 128);
}

cudaError_t attention_launch(const AttnParams& p, cudaStream_t s, bool pdl) {
  const int G = p.hq / p.hkv;
  if (p.d == 128) {
    if (G <= 4) return launch_attn<128, 4>(p, s, pdl);
    if (G == 8) return launch_attn<128, 8>(p, s, pdl);
  } else if (p.d == 64) {
    if (G <= 4) return launch_attn<64, 4>(p, s, pdl);
    if (G == 8) return launch_attn<64, 8>(p, s, pdl);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dflash
