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
#include "attention.cuh"

namespace dflash {

constexpr int kAttnBufs = 2;  // double-buffered 64-key chunks (measured best)

template <int D, int NW, int TERMS>
__global__ void __launch_bounds__(NW * 32) attn_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(128) uint8_t sm[];
  const int G = p.hq / p.hkv;
  const int R = 16 * NW / G;
  const int split = blockIdx.x, qt = blockIdx.y;
  const int req = blockIdx.z / p.hkv, g = blockIdx.z % p.hkv;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int group = lane / 4, tq = lane % 4;
  griddep_launch_dependents();
  griddep_wait();
  AttnAcc<D> acc;
  if (!attn_accumulate<D, NW, kAttnBufs, CtaSync, TERMS>(p, split, qt, req, g, tid, sm, CtaSync{}, acc))
    return;
  const float (&o)[D / 8][4] = acc.o;
  const float* m_r = acc.m;
  const float* l_r = acc.l;
  const int row_lo = acc.row_lo, head = acc.head;
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
        const size_t ob = ((static_cast<size_t>(req) * p.n + row) * p.hq + hd) * D;
#pragma unroll
        for (int t = 0; t < D / 32; ++t) {
          const float v = acc[t] * inv;
          const uint16_t hi = f2bf(v);
          p.out[ob + lane + 32 * t] = hi;
          if (p.out_lo != nullptr) p.out_lo[ob + lane + 32 * t] = bf16_lo_part(v, hi);
        }
      }
    }
    if (SC > 1) cluster_sync();  // peers may still read this CTA's partials until here
    return;
  }

  attn_store_partial<D>(p, split, req, acc, lane);
}

// One warp per (row, head): merge the splits that cover the row, in order.
// Lane s holds split s's (m, l) (splits in groups of 32); the O partials of a
// group are loaded together before they are accumulated in split order.
template <int D>
__global__ void __launch_bounds__(128) attn_combine_kernel(const __grid_constant__ AttnParams p) {
  griddep_launch_dependents();
  griddep_wait();
  const int vec = blockIdx.x * 4 + threadIdx.x / 32;
  if (vec >= p.batch * p.n * p.hq) return;
  attn_combine_vec<D>(p, vec, threadIdx.x % 32);
}

size_t attention_part_floats(int n_splits, int rows, int hq, int d) {
  return static_cast<size_t>(n_splits) * rows * hq * (d + 2);
}

template <int D, int NW, int TERMS>
static cudaError_t launch_attn(const AttnParams& p, cudaStream_t s, bool pdl) {
  static thread_local int attr_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<D, NW, TERMS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         attn_smem_bytes<D, kAttnBufs, TERMS>());
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_kernel<D, NW, TERMS>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_kernel<D, NW, TERMS>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
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
  cfg.dynamicSmemBytes = attn_smem_bytes<D, kAttnBufs, TERMS>();
  cfg.stream = s;
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  count_launch();
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_kernel<D, NW, TERMS>, p);
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

template <int TERMS>
static cudaError_t launch_terms(const AttnParams& p, cudaStream_t s, bool pdl) {
  const int G = p.hq / p.hkv;
  if (p.d == 128) {
    if (G <= 4) return launch_attn<128, 4, TERMS>(p, s, pdl);
    if (G == 8) return launch_attn<128, 8, TERMS>(p, s, pdl);
  } else if (p.d == 64) {
    if (G <= 4) return launch_attn<64, 4, TERMS>(p, s, pdl);
    if (G == 8) return launch_attn<64, 8, TERMS>(p, s, pdl);
  }
  return cudaErrorInvalidValue;
}

cudaError_t attention_launch(const AttnParams& p, cudaStream_t s, bool pdl) {
  return p.kv_terms == 2 ? launch_terms<2>(p, s, pdl) : launch_terms<1>(p, s, pdl);
}

}  // namespace dflash
