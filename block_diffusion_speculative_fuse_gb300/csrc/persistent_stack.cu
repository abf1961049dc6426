// Persistent layer-stack kernel for decode-sized draft steps (block rows +
// context rows <= 32): the whole drafter stack and the LM head in one launch,
// one CTA per SM, phases separated by grid barriers.
//
// Why: at batch 1 every GEMM of the stack streams 33-200 MB of weights in a
// few microseconds, and with one kernel per GEMM the HBM pipe drains at every
// kernel boundary.  Here the TMA producer warp walks the static list of all
// weight tiles this CTA will multiply, across phases and layers, and keeps the
// shared-memory ring full of the *next* GEMM's weights while the other warps
// finish reductions, attention and the grid barrier.  Only the (tiny)
// activation tile of a stage waits for the barrier that makes it valid.
//
// Roles (192 threads): warp 0 lane 0 = TMA producer; warp 1 = TMEM owner, lane
// 0 = MMA issuer (tcgen05.mma M=128 N=32 K=16, fp32 accumulators double
// buffered in TMEM); warps 2-5 = compute (drain accumulators, reductions,
// epilogues, attention, barriers).
//
// GEMM phases are stream-K: the phase's (tile, k-block) iterations are split
// evenly over the CTAs; each CTA writes an fp32 partial for every tile segment
// it covers, and the following reduce phase sums a tile's segments in order
// (deterministic) and runs the fused epilogue.  Per layer: QKV, reduce (q/k
// norm, RoPE, K/V routing), attention, combine, O, reduce (residual [+ block
// conv] + next-norm inputs), gate/up, reduce (SwiGLU), down, reduce (residual
// + next-norm inputs); then LM head, reduce (per-tile argmax), argmax.
//
// Launched cooperatively (all CTAs co-resident).  Every wait is bounded by
// %globaltimer: on timeout the status word gets DFLASH_ERR_TIMEOUT and the
// kernel runs to its end without waiting further.
#include "attention.cuh"
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace dflash {

namespace {

constexpr int kStages = 7;
constexpr int kBN = 32;                         // MMA N: activation rows, padded
constexpr int kA = kTileN * kTileK * 2;         // 16 KB weight tile
constexpr int kB = kBN * kTileK * 2;            // 4 KB activation tile
constexpr int kStageBytes = kA + kB;
constexpr int kRing = kStages * kStageBytes;    // 160 KB
constexpr int kWork = 66 * 1024;                // attention K/V buffers + page ids, or staged tile
constexpr int kCtl = 2048;                      // barriers, TMEM slot, row scales, routing
constexpr int kSmem = kRing + kWork + kCtl + 1024;
constexpr int kThreads = 192;
constexpr int kTmemCols = 64;                   // two 32-column accumulators

enum Kind : int {
  K_QKV_G = 0, K_QKV_R, K_ATT, K_COMB, K_O_G, K_O_R, K_GU_G, K_GU_R, K_DN_G, K_DN_R,
  kPerLayer,
  K_LM_G = 100, K_LM_R, K_ARG
};

__device__ __forceinline__ int phase_kind(int phi, int L, int* layer) {
  if (phi < L * kPerLayer) {
    *layer = phi / kPerLayer;
    return phi % kPerLayer;
  }
  *layer = L;
  return K_LM_G + (phi - L * kPerLayer);
}
__device__ __forceinline__ bool is_gemm(int k) {
  return k == K_QKV_G || k == K_O_G || k == K_GU_G || k == K_DN_G || k == K_LM_G;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

}  // namespace

struct GemmGeo {
  const CUtensorMap* w;
  const CUtensorMap* x;
  int w_row0, tile_step, half_gap, n_tiles, kbt, M;
};

__device__ __forceinline__ GemmGeo gemm_geo(const PersistParams& P, int kind, int l) {
  GemmGeo g;
  g.tile_step = kTileN;
  g.half_gap = 64;
  switch (kind) {
    case K_QKV_G:
      g.w = &P.m_wqkv; g.x = &P.x_a; g.w_row0 = l * P.qkv_rows; g.n_tiles = P.qkv_rows / kTileN;
      g.kbt = P.H / kTileK; g.M = P.M_qkv;
      break;
    case K_O_G:
      g.w = &P.m_wo; g.x = &P.x_o; g.w_row0 = l * P.H; g.n_tiles = P.H / kTileN;
      g.kbt = P.q_dim / kTileK; g.M = P.nb;
      break;
    case K_GU_G:
      g.w = &P.m_gu; g.x = &P.x_a2; g.w_row0 = l * 2 * P.F; g.tile_step = 64; g.half_gap = P.F;
      g.n_tiles = 2 * P.F / kTileN; g.kbt = P.H / kTileK; g.M = P.nb;
      break;
    case K_DN_G:
      g.w = &P.m_down; g.x = &P.x_h; g.w_row0 = l * P.H; g.n_tiles = P.H / kTileN;
      g.kbt = P.F / kTileK; g.M = P.nb;
      break;
    default:  // K_LM_G
      g.w = &P.m_lm; g.x = &P.x_a2; g.w_row0 = 0; g.n_tiles = P.V / kTileN;
      g.kbt = P.H / kTileK; g.M = P.nb;
      break;
  }
  return g;
}

// stream-K partition of a phase's n_tiles*kbt iterations over `nc` CTAs
__device__ __forceinline__ long long sk_lo(long long total, int c, int nc) {
  return total * c / nc;
}
// CTA whose range holds iteration i
__device__ __forceinline__ int sk_owner(long long total, long long i, int nc) {
  return static_cast<int>(((i + 1) * nc - 1) / total);
}

// Upper bound of the segments a tile of this phase is split into.
__device__ __forceinline__ int segs_bound(const GemmGeo& g, int nc) {
  const long long total = static_cast<long long>(g.n_tiles) * g.kbt;
  return static_cast<int>((static_cast<long long>(g.kbt) * nc + total - 1) / total) + 1;
}
__device__ __forceinline__ float* part_slot(const PersistParams& P, const GemmGeo& g, int nc,
                                            int tile, int seg) {
  return P.part + (static_cast<size_t>(tile) * segs_bound(g, nc) + seg) * (kBN * kTileN);
}

// Grid barrier over the compute warps of all CTAs; counter target is monotonic.
__device__ __forceinline__ void grid_sync(const PersistParams& P, unsigned target, int ltid) {
  asm volatile("fence.proxy.async.global;" ::: "memory");
  GroupSync{1}();
  if (ltid == 0) {
    __threadfence();
    atomicAdd(P.bar, 1u);
    const uint64_t t0 = global_ns();
    while (ld_acquire(P.bar) < target) {
      if (*reinterpret_cast<volatile int*>(P.status) != 0) break;  // another wait gave up
      if (global_ns() - t0 > kWaitLimitNs) {
        raise_status(P.status, DFLASH_ERR_TIMEOUT, 401);
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
  }
  GroupSync{1}();
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    persistent_stack_kernel(const __grid_constant__ PersistParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* work = smem + kRing;
  uint8_t* ctl = work + kWork;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctl);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  float* rinv = reinterpret_cast<float*>(ctl + 512);
  int* route = reinterpret_cast<int*>(ctl + 512 + kBN * 4);

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int nc = gridDim.x, cta = blockIdx.x;
  const int L = P.n_layers;
  const int n_phases = L * kPerLayer + 3;
  // any wait that gives up records a status; every other wait then stops too
  volatile int* abort_flag = reinterpret_cast<volatile int*>(P.status);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 128);
    }
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();
      int pend_s[kStages], pend_k[kStages], pend_phi[kStages];
      const CUtensorMap* pend_x[kStages];
      int np = 0, it = 0;
      int ready_phi = 0;  // phases <= ready_phi have their activations written
      bool dead = false;
      // Poll the barrier counter and issue the activation loads that became
      // valid.  Called only while blocked (full ring) or draining, so the
      // steady-state stream issues no global loads.
      auto service = [&]() {
        if (np == 0) return;
        const unsigned c = ld_acquire(P.bar);
        ready_phi = static_cast<int>(c / static_cast<unsigned>(nc));
        int k = 0;
        while (k < np && pend_phi[k] <= ready_phi) ++k;
        if (k == 0) return;
        asm volatile("fence.proxy.async.global;" ::: "memory");
        for (int i = 0; i < k; ++i)
          tma_load_2d(smem + kStages * kA + pend_s[i] * kB, pend_x[i], pend_k[i], 0,
                      &full[pend_s[i]], pol_x);
        for (int i = k; i < np; ++i) {
          pend_s[i - k] = pend_s[i];
          pend_k[i - k] = pend_k[i];
          pend_phi[i - k] = pend_phi[i];
          pend_x[i - k] = pend_x[i];
        }
        np -= k;
      };
      for (int phi = 0; phi < n_phases && !dead; ++phi) {
        int l;
        const int kind = phase_kind(phi, L, &l);
        if (!is_gemm(kind)) continue;
        const GemmGeo g = gemm_geo(P, kind, l);
        const long long total = static_cast<long long>(g.n_tiles) * g.kbt;
        const long long lo = sk_lo(total, cta, nc), hi = sk_lo(total, cta + 1, nc);
        for (long long i = lo; i < hi && !dead; ++i, ++it) {
          const int tile = static_cast<int>(i / g.kbt), kb = static_cast<int>(i % g.kbt);
          const int s = it % kStages;
          if (it >= kStages) {
            const uint32_t ph = ((it / kStages) & 1) ^ 1;
            const uint32_t a = smem_u32(&empty[s]);
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(a, ph)) {
              service();
              if (*reinterpret_cast<volatile int*>(P.status) != 0) {
                dead = true;
                break;
              }
              if (global_ns() - t0 > kWaitLimitNs) {
                raise_status(P.status, DFLASH_ERR_TIMEOUT, 402);
                dead = true;
                break;
              }
            }
            if (dead) break;
          }
          const int kx = kb * kTileK;
          const int wrow = g.w_row0 + tile * g.tile_step;
          mbar_arrive_expect_tx(&full[s], kStageBytes);
          tma_load_2d(smem + s * kA, g.w, kx, wrow, &full[s], pol_w);
          tma_load_2d(smem + s * kA + kA / 2, g.w, kx, wrow + g.half_gap, &full[s], pol_w);
          if (np == 0 && phi <= ready_phi) {
            tma_load_2d(smem + kStages * kA + s * kB, g.x, kx, 0, &full[s], pol_x);
          } else {
            pend_s[np] = s;
            pend_k[np] = kx;
            pend_phi[np] = phi;
            pend_x[np] = g.x;
            ++np;
          }
        }
      }
      const uint64_t t0 = global_ns();
      while (np > 0 && !dead) {
        service();
        if (*reinterpret_cast<volatile int*>(P.status) != 0) break;
        if (global_ns() - t0 > kWaitLimitNs) {
          raise_status(P.status, DFLASH_ERR_TIMEOUT, 403);
          break;
        }
        __nanosleep(32);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = umma_idesc_bf16(kTileN, kBN);
      int it = 0, seg = 0;
      bool dead = false;
      for (int phi = 0; phi < n_phases && !dead; ++phi) {
        int l;
        const int kind = phase_kind(phi, L, &l);
        if (!is_gemm(kind)) continue;
        const GemmGeo g = gemm_geo(P, kind, l);
        const long long total = static_cast<long long>(g.n_tiles) * g.kbt;
        const long long lo = sk_lo(total, cta, nc), hi = sk_lo(total, cta + 1, nc);
        long long i = lo;
        while (i < hi && !dead) {
          const long long tile_end = (i / g.kbt + 1) * g.kbt;
          const long long end = hi < tile_end ? hi : tile_end;
          const int buf = seg & 1;
          if (!mbar_wait(&tempty[buf], ((seg >> 1) & 1) ^ 1, abort_flag)) {
            raise_status(P.status, DFLASH_ERR_TIMEOUT, 404);
            dead = true;
            break;
          }
          tc_fence_after();
          const uint32_t acc = tmem + buf * kBN;
          for (long long j = i; j < end; ++j, ++it) {
            const int s = it % kStages;
            if (!mbar_wait(&full[s], (it / kStages) & 1, abort_flag)) {
              raise_status(P.status, DFLASH_ERR_TIMEOUT, 405);
              dead = true;
              break;
            }
            tc_fence_after();
            const uint64_t ad = umma_desc_sw128(smem_u32(smem + s * kA));
            const uint64_t bd = umma_desc_sw128(smem_u32(smem + kStages * kA + s * kB));
#pragma unroll
            for (int k = 0; k < kTileK / 16; ++k)
              umma_bf16(acc, ad + 2 * k, bd + 2 * k, idesc, (j > i || k > 0) ? 1u : 0u);
            umma_commit(&empty[s]);
          }
          umma_commit(&tfull[buf]);
          ++seg;
          i = end;
        }
      }
    }
  } else {
    // ------------------------------------------------ compute warps
    const int ltid = tid - 64;         // 0..127
    const int cw = ltid / 32;          // compute warp 0..3
    const int quad = warp & 3;         // TMEM lane quadrant of this warp
    const GroupSync gsync{1};
    int seg = 0;
    for (int phi = 0; phi < n_phases; ++phi) {
      int l;
      const int kind = phase_kind(phi, L, &l);
      if (is_gemm(kind)) {
        const GemmGeo g = gemm_geo(P, kind, l);
        const long long total = static_cast<long long>(g.n_tiles) * g.kbt;
        const long long lo = sk_lo(total, cta, nc), hi = sk_lo(total, cta + 1, nc);
        long long i = lo;
        while (i < hi) {
          const int tile = static_cast<int>(i / g.kbt);
          const long long tile_end = (tile + 1LL) * g.kbt;
          const long long end = hi < tile_end ? hi : tile_end;
          const int sidx = cta - sk_owner(total, static_cast<long long>(tile) * g.kbt, nc);
          const int buf = seg & 1;
          const bool ok = mbar_wait(&tfull[buf], (seg >> 1) & 1, abort_flag);
          if (!ok && ltid == 0) raise_status(P.status, DFLASH_ERR_TIMEOUT, 406);
          tc_fence_after();
          float* dst = part_slot(P, g, nc, tile, sidx);
          const int f = quad * 32 + lane;
#pragma unroll
          for (int c = 0; c < kBN / 16; ++c) {
            float v[16];
            tmem_ld16(tmem + buf * kBN + (static_cast<uint32_t>(quad * 32) << 16) + c * 16, v);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c * 16 + j < g.M) dst[(c * 16 + j) * kTileN + f] = v[j];
          }
          tc_fence_before();
          mbar_arrive(&tempty[buf]);
          ++seg;
          i = end;
        }
      } else if (kind == K_ATT) {
        const AttnParams& a = P.att;
        AttnParams ap = a;
        ap.pool = P.pool + P.pool_layer_elems * l;
        const int G = a.hq / a.hkv;
        const int R = 64 / G;
        const int n_qt = (a.n + R - 1) / R;
        const int units = a.batch * a.hkv * n_qt * a.n_splits;
        for (int u = cta; u < units; u += nc) {
          const int split = u % a.n_splits;
          int r = u / a.n_splits;
          const int qt = r % n_qt;
          r /= n_qt;
          const int g = r % a.hkv, req = r / a.hkv;
          AttnAcc<D> acc;
          if (attn_accumulate<D, 4, 2>(ap, split, qt, req, g, ltid, work, gsync, acc))
            attn_store_partial<D>(ap, split, req, acc, lane);
          gsync();  // the K/V buffers are reused by the next unit
        }
      } else if (kind == K_COMB) {
        const AttnParams& a = P.att;
        const int nvec = a.batch * a.n * a.hq;
        for (int v = cta * 4 + cw; v < nvec; v += nc * 4) {
          attn_combine_vec<D>(a, v, lane);
        }
      } else if (kind == K_ARG) {
        // one warp per row: (max, lowest index) over the LM-head tile maxima
        const int n_tiles = P.V / kTileN;
        for (int row = cta * 4 + cw; row < P.nb; row += nc * 4) {
          const int i = row % P.block;
          if (i == 0) continue;
          float bv = -INFINITY;
          int bi = 0x7fffffff;
          for (int t = lane; t < n_tiles; t += 32) {
            const float v = __ldcg(P.amax_val + static_cast<size_t>(row) * n_tiles + t);
            const int j = __ldcg(P.amax_idx + static_cast<size_t>(row) * n_tiles + t);
            if (v > bv || (v == bv && j < bi)) { bv = v; bi = j; }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
          }
          if (lane == 0) P.draft[(row / P.block) * (P.block - 1) + i - 1] = bi;
        }
      } else {
        // reduce phases: sum the tile's segments in order, then the epilogue
        const int gk = kind == K_LM_R ? K_LM_G : kind - 1;
        const GemmGeo g = gemm_geo(P, gk, l);
        const long long total = static_cast<long long>(g.n_tiles) * g.kbt;
        GemmParams ep = P.ep;
        ep.M = g.M;
        ep.N = g.n_tiles * kTileN;
        const int H = P.H;
        const float* ssq_in = nullptr;
        int norm_rows = g.M;
        switch (kind) {
          case K_QKV_R:
            ep.mode = EPI_QKV;
            if (P.ep.qkv.q_norm != nullptr) {
              ep.qkv.q_norm = P.ep.qkv.q_norm + static_cast<size_t>(l) * P.head_dim;
              ep.qkv.k_norm = P.ep.qkv.k_norm + static_cast<size_t>(l) * P.head_dim;
            }
            ep.qkv.pool = P.pool + P.pool_layer_elems * l;
            ssq_in = P.ssq_a;
            norm_rows = P.nb;
            break;
          case K_O_R:
            ep.mode = EPI_RESID;
            ep.gnext = P.post_norm + static_cast<size_t>(l) * H;
            ep.xg_out = P.a2;
            ep.ssq_out = P.ssq_a2;
            if (P.conv != nullptr && P.conv_width > 0) {
              ep.conv = P.conv + static_cast<size_t>(l) * H * P.conv_width;
              ep.conv_width = P.conv_width;
            }
            break;
          case K_GU_R:
            ep.mode = EPI_SWIGLU;
            ep.out = P.hmid;
            ep.ld_out = P.F;
            ssq_in = P.ssq_a2;
            break;
          case K_DN_R: {
            const bool last = (l == L - 1);
            ep.mode = EPI_RESID;
            ep.gnext = last ? P.final_norm : P.in_norm + static_cast<size_t>(l + 1) * H;
            ep.xg_out = last ? P.a2 : P.a;
            ep.ssq_out = last ? P.ssq_a2 : P.ssq_a;
            break;
          }
          default:  // K_LM_R
            ep.mode = EPI_ARGMAX;
            ssq_in = P.logits != nullptr ? P.ssq_a2 : nullptr;
            break;
        }
        float* ts = reinterpret_cast<float*>(work);
        for (int tile = cta; tile < g.n_tiles; tile += nc) {
          const long long first = static_cast<long long>(tile) * g.kbt;
          const int c0 = sk_owner(total, first, nc);
          const int nseg = sk_owner(total, first + g.kbt - 1, nc) - c0 + 1;
          // sum segments in order: thread owns float4 chunks of the tile
          for (int c = ltid; c < g.M * 32; c += 128) {
            const int r = c / 32, c4 = c % 32;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int sg = 0; sg < nseg; ++sg) {
              const float4 v = __ldcg(reinterpret_cast<const float4*>(part_slot(P, g, nc, tile, sg) + r * kTileN) + c4);
              acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
            }
            *reinterpret_cast<float4*>(ts + r * kTsLd + c4 * 4) = acc;
          }
          gsync();
          if (ssq_in != nullptr) {
            for (int r = cw; r < g.M; r += 4) {
              const float* q = ssq_in + static_cast<size_t>(r) * (H / kTileN);
              float ss = 0.f;
              for (int t = lane; t < H / kTileN; t += 32) ss += __ldcg(q + t);  // written by other CTAs
              ss = warp_sum(ss);
              if (lane == 0) rinv[r] = r < norm_rows ? rsqrtf(ss / static_cast<float>(H) + P.eps) : 1.f;
            }
            gsync();
            for (int idx = ltid; idx < g.M * kTileN; idx += 128) ts[(idx / kTileN) * kTsLd + idx % kTileN] *= rinv[idx / kTileN];
            gsync();
          }
          switch (kind) {
            case K_QKV_R: epi_qkv(ep, ts, tile, 0, g.M, route, kBN, ltid, gsync); break;
            case K_O_R:
            case K_DN_R: epi_resid(ep, ts, tile, 0, g.M, ltid, gsync); break;
            case K_GU_R: epi_swiglu(ep, ts, tile, 0, g.M, ltid, gsync); break;
            default: epi_argmax(ep, ts, tile, 0, g.M, ltid, gsync, g.n_tiles); break;
          }
          gsync();
        }
      }
      if (phi + 1 < n_phases) grid_sync(P, static_cast<unsigned>(phi + 1) * nc, ltid);
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

int persistent_smem_bytes() { return kSmem; }

// CTAs of the persistent launch: at most one per SM, and no more than the
// smallest GEMM phase has (tile, k-block) iterations, so that every CTA owns at
// least one iteration of every phase (the segment numbering relies on it).
int persistent_ctas(const PersistParams& p, int sms) {
  const long long tot[5] = {static_cast<long long>(p.qkv_rows / kTileN) * (p.H / kTileK),
                            static_cast<long long>(p.H / kTileN) * (p.q_dim / kTileK),
                            static_cast<long long>(2 * p.F / kTileN) * (p.H / kTileK),
                            static_cast<long long>(p.H / kTileN) * (p.F / kTileK),
                            static_cast<long long>(p.V / kTileN) * (p.H / kTileK)};
  long long n = sms;
  for (long long t : tot) n = n < t ? n : t;
  return static_cast<int>(n);
}

// Largest tiles x segment-bound product over the GEMM phases (partial slots).
size_t persistent_part_floats(const PersistParams& p, int nc) {
  struct Ph { long long n_tiles, kbt; };
  const Ph ph[5] = {{p.qkv_rows / kTileN, p.H / kTileK}, {p.H / kTileN, p.q_dim / kTileK},
                    {2LL * p.F / kTileN, p.H / kTileK}, {p.H / kTileN, p.F / kTileK},
                    {p.V / kTileN, p.H / kTileK}};
  long long mx = 0;
  for (const Ph& q : ph) {
    const long long total = q.n_tiles * q.kbt;
    const long long segs = (q.kbt * nc + total - 1) / total + 1;
    mx = mx > q.n_tiles * segs ? mx : q.n_tiles * segs;
  }
  return static_cast<size_t>(mx) * kBN * kTileN;
}

template <int D>
static cudaError_t persistent_launch_d(const PersistParams& p, int n_ctas, cudaStream_t s) {
  static thread_local int attr_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(persistent_stack_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(persistent_stack_kernel<D>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_device = dev;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_ctas, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launch();
  return cudaLaunchKernelEx(&cfg, persistent_stack_kernel<D>, p);
}

cudaError_t persistent_launch(const PersistParams& p, int n_ctas, cudaStream_t s) {
  return p.head_dim == 128 ? persistent_launch_d<128>(p, n_ctas, s)
                           : persistent_launch_d<64>(p, n_ctas, s);
}

}  // namespace dflash
