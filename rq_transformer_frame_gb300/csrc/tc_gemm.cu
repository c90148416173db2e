// tc_gemm.cu -- weights x batch on the tcgen05 tensor cores (batch 2..64, padded to a
// multiple of 16).
//
// At batch B the linears of a frame become Y[b][n] = sum_k X[b][k] W[n][k], a real dense
// contraction (B flops per weight byte... still below the tensor ridge, so the kernel
// stays bound by streaming W once).  One CTA owns a 128-row tile of W (or 64 gate + 64
// multiplier rows for the SiLU-gated layers) and a range of 64-wide K steps:
//   warp 0 (one lane)  TMA: W tile box {64, 128} and X box {64, NB} per K step, 128-byte
//                      swizzle, into a ring of shared-memory stages (mbarrier tx count);
//   warp 1             allocates NB tensor-memory columns; one lane issues 4
//                      tcgen05.mma.kind::f16 (M 128, N NB, K 16) per stage and commits
//                      each stage back to its "empty" barrier;
//   warps 2-5          read the 128 x NB f32 accumulator from tensor memory
//                      (tcgen05.ld, one lane = one W row) and run the fused epilogue.
// With split-K, from 32 sessions on, the splits of a tile run as one thread-block
// cluster: each stores its partial tile in its own shared memory, and after a cluster
// barrier split r adds every split's partial (distributed shared memory, in split order --
// deterministic) for the 16-session chunks r, r + splits, ... and runs their epilogue, so
// the merge needs no round trip to L2 and the epilogue is spread over the splits.  At 16
// sessions (one chunk) each split stores its partial tile to L2 and the last one to finish
// (atomic ticket) adds them in split order and runs the epilogue.
#include "tc_epilogue.cuh"

namespace rqk {
namespace tcg {

template <int NB>
__global__ void __launch_bounds__(kThreads, 2)
    tc_gemm_kernel(const TcParams p, const __grid_constant__ CUtensorMap wmap,
                   const __grid_constant__ CUtensorMap xmap) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t s_full[8], s_empty[8], s_done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_last;
  __shared__ volatile int s_abort;
  __shared__ int s_issued, s_consumed;
  __shared__ EpiShared s_epi;
  constexpr int kN = kOpndParts * NB;  // MMA columns: the bf16 parts of each session
  constexpr uint32_t kCols = kN <= 64 ? 64u : (kN <= 128 ? 128u : 256u);  // power of two
  const TcPlan& pl = p.pl;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NS = pl.n_stages;
  constexpr int kBBytes = kN * kBK * 2;
  constexpr int kStage = kABytes + kBBytes;  // both multiples of 1024
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tile = blockIdx.x / pl.splits, split = blockIdx.x % pl.splits;
  const int ks0 = split * pl.ksteps_split;
  const int ks1 = min(ks0 + pl.ksteps_split, pl.ksteps);
  const int nk = ks1 - ks0;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], 1);
    }
    mbar_init(&s_done, 1);
    fence_barrier_init();
    s_abort = 0;
    s_issued = 0;
    s_consumed = 0;
    tc::prefetch_tmap(&wmap);
    tc::prefetch_tmap(&xmap);
  }
  if (warp == 1) {
    tc::tmem_alloc(&s_tmem, kCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();  // weights: read once per frame
      const uint64_t pol_x = l2_policy_evict_last();  // operands: read by every tile
      const int row_a = pl.paired ? tile * 64 : tile * kBM;
      auto load_w = [&](int i) {
        uint8_t* a = smem + (size_t)(i % NS) * kStage;
        const int kx = (ks0 + i) * kBK;
        tc::tma_load_2d(a, &wmap, kx, row_a, &s_full[i % NS], pol);
        if (pl.paired)
          tc::tma_load_2d(a + kABytes / 2, &wmap, kx, pl.n_out + row_a, &s_full[i % NS], pol);
      };
      auto load_x = [&](int i) {
        uint8_t* b = smem + (size_t)(i % NS) * kStage + kABytes;
        tc::tma_load_2d(b, &xmap, (ks0 + i) * kBK, 0, &s_full[i % NS], pol_x);
      };
      // the weights do not depend on the previous kernel: stream the first stages now,
      // the activations once that kernel has finished
      const int pre = min(NS, nk);
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&s_full[i], (uint32_t)kStage);
        load_w(i);
      }
      pdl_wait();
      for (int i = 0; i < pre; ++i) load_x(i);
      int i = pre;
      for (; i < nk; ++i) {
        const int s = i % NS;
        if (!mbar_wait(&s_empty[s], (uint32_t)((i / NS) - 1) & 1u)) {
          atomicOr(p.status, kDevTimeout);
          s_abort = 1;
          break;
        }
        mbar_arrive_expect_tx(&s_full[s], (uint32_t)kStage);
        load_w(i);
        load_x(i);
      }
      s_issued = i;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(kBM, kN);
      for (int i = 0; i < nk; ++i) {
        const int s = i % NS;
        if (s_abort || !mbar_wait(&s_full[s], (uint32_t)(i / NS) & 1u)) {
          atomicOr(p.status, kDevTimeout);
          s_abort = 1;
          break;
        }
        tc::fence_after_sync();
        const uint32_t a = smem_u32(smem + (size_t)s * kStage);
        const uint32_t b = a + kABytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          tc::mma_bf16(tmem, tc::sw128_desc(a + kk * 32), tc::sw128_desc(b + kk * 32), idesc,
                       (i > 0 || kk > 0) ? 1u : 0u);
        tc::commit(&s_empty[s]);
        s_consumed = i + 1;
      }
      tc::commit(&s_done);  // after every MMA issued above (also on abort)
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue warps
    pdl_wait();
    const int q = warp & 3;  // tensor-memory lane quarter this warp may read
    const int m = q * 32 + lane;
    const int et = tid - 64;  // 0..127 among the epilogue warps
    // K splits: the CTAs of a tile form one cluster; split r (its rank) finishes the
    // 16-session chunks r, r + splits, ... from every split's partial in the cluster's
    // shared memory, in split order (deterministic)
    const int S = pl.splits;
    // (compile time: the 16-session instantiation keeps only the L2 merge, the others only
    // the cluster one; the host plans the same split)
    constexpr bool kClu = NB >= 32;
    const bool clu = kClu && S > 1;
    const int c0f = clu ? 16 * split : 0;  // this CTA's first chunk
    const int cstep = clu ? 16 * S : 16;
    // while the MMAs run: the fused-RMSNorm scales, and the old residual values of the
    // first chunk
    if (p.ss_in && et < NB) {
      float ss = 0.f;
      for (int t = 0; t < p.ss_tiles; ++t) ss += p.ss_in[(size_t)t * NB + et];
      s_epi.inv[et] = 1.0f / sqrtf(p.eps + ss / (float)p.rms_K);
    }
    float old0[16];
    {
      const int row = tile * kBM + m;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        old0[i] = (p.epi == EPI_RESID && !pl.paired && row < pl.n_out && c0f + i < p.B)
                      ? p.out[(size_t)(c0f + i) * p.out_bs + row]
                      : 0.f;
    }
    if (!mbar_wait(&s_done, 0u)) s_abort = 1;
    bar_sync(1, 128);
    const bool ok = !s_abort;  // the same for all epilogue threads
    tc::fence_after_sync();
    if (!ok) atomicOr(p.status, kDevTimeout);
    // this split's accumulator into its shared memory as [NB][kBM] f32 (the stages are
    // free: every MMA, hence every load into them, has completed)
    float* part_s = reinterpret_cast<float*>(smem);
    if (kClu && clu && ok) {
#pragma unroll
      for (int c0 = 0; c0 < NB; c0 += 16) {
        float v[16];
        load_sum3<NB>(tmem + ((uint32_t)(q * 32) << 16), c0, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) part_s[(size_t)(c0 + i) * kBM + m] = v[i];
      }
    }
    if (kClu && clu) tc::cluster_sync();  // every split's partial written
    bool run = ok;
    if (!kClu && S > 1 && ok) {
      // store this split's partial, then the last split of the tile merges in order
      float* mine = p.partial + ((size_t)(tile * S + split) * NB) * kBM;
#pragma unroll
      for (int c0 = 0; c0 < NB; c0 += 16) {
        float v[16];
        load_sum3<NB>(tmem + ((uint32_t)(q * 32) << 16), c0, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) mine[(size_t)(c0 + i) * kBM + m] = v[i];
      }
      __threadfence();
      bar_sync(1, 128);
      if (et == 0) s_last = (atomicAdd(&p.tickets[tile], 1) == S - 1);
      bar_sync(1, 128);
      run = s_last != 0;
      if (run) __threadfence();
    }
    if (run) {
      const uint32_t part_a = smem_u32(part_s);
#pragma unroll 1
      for (int c0 = c0f; c0 < NB; c0 += cstep) {
        // the residual's old values of this CTA's next chunk load while this one runs
        float old1[16];
        {
          const int row = tile * kBM + m;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            old1[i] = (p.epi == EPI_RESID && !pl.paired && row < pl.n_out && c0 + cstep + i < p.B)
                          ? p.out[(size_t)(c0 + cstep + i) * p.out_bs + row]
                          : 0.f;
        }
        float v[16];
        if (kClu && clu) {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = 0.f;
          for (int r = 0; r < S; ++r) {
            float a[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              a[i] = tc::ld_cluster(
                  tc::mapa(part_a + (uint32_t)(((c0 + i) * kBM + m) * 4), (uint32_t)r));
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] += a[i];
          }
        } else if (!kClu && S > 1) {
          // splits added in split order; the loads of up to four splits are issued before
          // their adds, one round trip to L2 for up to four partials
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = 0.f;
          const size_t sstride = (size_t)NB * kBM;  // floats between splits of a tile
          const float* src = p.partial + ((size_t)tile * S * NB + c0) * kBM + m;
          for (int sp = 0; sp < S; sp += 4) {
            float a[4][16];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
              for (int i = 0; i < 16; ++i)
                a[u][i] = sp + u < S ? __ldcg(src + (size_t)(sp + u) * sstride + (size_t)i * kBM)
                                     : 0.f;
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (sp + u < S) {
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] += a[u][i];
              }
          }
        } else {
          load_sum3<NB>(tmem + ((uint32_t)(q * 32) << 16), c0, v);
        }
        if (p.ss_in) {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] *= s_epi.inv[c0 + i];
        }
        epilogue_chunk(p, v, c0, tile, m, lane, q, s_epi, old0);
#pragma unroll
        for (int i = 0; i < 16; ++i) old0[i] = old1[i];
        if (p.ss_out) {
          bar_sync(1, 128);
          if (et < 16) {
            const float ss = s_epi.ss[0][c0 + et] + s_epi.ss[1][c0 + et] +
                             s_epi.ss[2][c0 + et] + s_epi.ss[3][c0 + et];
            p.ss_out[(size_t)tile * NB + c0 + et] = ss;
          }
        }
      }
      if (p.epi == EPI_ARGMAX) {
        bar_sync(1, 128);
        // the sessions of this CTA's chunks
        if (et < NB && et < p.B && (!clu || ((et >> 4) % S) == split)) {
          unsigned long long k = s_epi.key[0][et];
          for (int w = 1; w < 4; ++w) k = s_epi.key[w][et] > k ? s_epi.key[w][et] : k;
          atomicMax(p.keys + (size_t)et * 9 + p.key_index, k);
        }
      }
    }
    if (!kClu && S > 1 && run && et == 0) p.tickets[tile] = 0;
    tc::fence_before_sync();
    if (kClu && clu) tc::cluster_sync();  // this CTA's partial stays until every split read it
  }
  if (NB >= 32 && warp < 2 && pl.splits > 1) {
    // the producer and MMA warps take part in the cluster's two barriers
    tc::cluster_sync();
    tc::cluster_sync();
  }
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kCols);
  }
  if (s_abort && tid == 0) {
    // wind down: wait (bounded) for TMA loads that no MMA consumed
    for (int i = s_consumed; i < s_issued; ++i)
      (void)mbar_wait(&s_full[i % NS], (uint32_t)(i / NS) & 1u);
  }
}

}  // namespace tcg
}  // namespace rqk

// ---------------------------------------------------------------- activation prep
namespace rqk {
namespace tcg {

// one CTA per padded session row: xb[.][b] = bf16 parts of (in[b] (* alpha * 1/sqrt(eps +
// mean(in^2)))) ("moshi_lm.rs", `rms_norm`), zero rows for b >= B; side[b] = the f32 result
__global__ void __launch_bounds__(256) prep_bf16_kernel(const float* in, long long in_bs,
                                                        const float* alpha, float eps, int B,
                                                        int K, uint16_t* xb, float* side,
                                                        long long side_bs) {
  __shared__ float s_red[8];
  const int b = blockIdx.x, tid = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  const size_t ps = (size_t)gridDim.x * K;  // operand part stride
  if (b >= B) {
    for (int k = tid; k < K; k += 256) store_bf16_parts(xb, ps, (size_t)b * K + k, 0.f);
    return;
  }
  const float* x = in + (size_t)b * in_bs;
  float inv = 1.f;
  if (alpha) {
    float ss = 0.f;
    for (int k = tid; k < K; k += 256) ss = fmaf(x[k], x[k], ss);
    ss = warp_sum(ss);
    if ((tid & 31) == 0) s_red[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < 8; ++w) tot += s_red[w];
    inv = 1.0f / sqrtf(eps + tot / (float)K);
  }
  for (int k = tid; k < K; k += 256) {
    const float v = alpha ? x[k] * alpha[k] * inv : x[k];
    store_bf16_parts(xb, ps, (size_t)b * K + k, v);
    if (side) side[(size_t)b * side_bs + k] = v;
  }
}

}  // namespace tcg

cudaError_t launch_prep_bf16(const float* in, long long in_bs, const float* alpha, float eps,
                             int B, int NB, int K, uint16_t* xb, float* side, long long side_bs,
                             cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)NB, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, tcg::prep_bf16_kernel, in, in_bs, alpha, eps, B, K, xb, side,
                            side_bs);
}

// ---------------------------------------------------------------- host side
TcPlan plan_tc(int n_out, int K, int NB, bool paired, int num_sms) {
  TcPlan pl{};
  pl.n_out = n_out;
  pl.K = K;
  pl.NB = NB;
  pl.paired = paired ? 1 : 0;
  const int rows = paired ? 64 : tcg::kBM;
  pl.tiles_m = (n_out + rows - 1) / rows;
  pl.ksteps = K / tcg::kBK;
  // split K so the grid fills at most one wave of 2 CTAs per SM (a partial second wave
  // would idle most SMs for its duration), keeping >= 4 K steps per split
  int splits = (2 * num_sms) / pl.tiles_m;
  const int max_splits = pl.ksteps / 4 > 0 ? pl.ksteps / 4 : 1;
  if (splits > max_splits) splits = max_splits;
  // at 64 columns a split's partial tile is 32 KB and beyond four splits merging them
  // costs more than the extra CTAs return (measured on out_proj / gate_out)
  if (NB >= 64 && splits > 4) splits = 4;
  // from 32 sessions (two or more 16-session chunks) the splits of a tile form one
  // thread-block cluster (portable size: at most 8); at 16 the L2 merge measured faster
  pl.cluster = NB >= 32 ? 1 : 0;
  if (pl.cluster && splits > 8) splits = 8;
  if (splits < 1) splits = 1;
  pl.ksteps_split = (pl.ksteps + splits - 1) / splits;
  pl.splits = (pl.ksteps + pl.ksteps_split - 1) / pl.ksteps_split;
  // two CTAs per SM: ~104 KB of dynamic shared memory each; a grid that fits one CTA per
  // SM (the small depformer GEMMs) takes up to ~200 KB, enough to have all of a CTA's
  // K steps in flight at once
  const int stage = tcg::kABytes + kOpndParts * NB * tcg::kBK * 2;
  const bool one_per_sm = pl.tiles_m * pl.splits <= num_sms;
  // (two per SM: 2 x (dynamic + ~11.5 KB static + 1 KB reserved) within 228 KB)
  int ns = ((one_per_sm ? 190 : 100) * 1024) / stage;  // + 1 KB alignment
  ns = ns < 2 ? 2 : (ns > 8 ? 8 : ns);
  if (one_per_sm && ns > pl.ksteps_split) ns = pl.ksteps_split < 2 ? 2 : pl.ksteps_split;
  pl.n_stages = ns;
  pl.smem = ns * stage + 1024;
  pl.bytes = (double)n_out * (paired ? 2.0 : 1.0) * K * 2.0;
  return pl;
}

template <int NB>
static cudaError_t launch_nb(const TcParams& p, const CUtensorMap& w, const CUtensorMap& x,
                             cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.pl.tiles_m * p.pl.splits), 1, 1);
  cfg.blockDim = dim3(tcg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)p.pl.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (p.pl.splits > 1 && p.pl.cluster) {  // the K splits of a tile form one cluster
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)p.pl.splits;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = (unsigned)n;
  return cudaLaunchKernelEx(&cfg, tcg::tc_gemm_kernel<NB>, p, w, x);
}

cudaError_t launch_tc(const TcParams& p, const CUtensorMap& wmap, const CUtensorMap& xmap,
                      cudaStream_t s, bool pdl) {
  switch (p.pl.NB) {
    case 16: return launch_nb<16>(p, wmap, xmap, s, pdl);
    case 32: return launch_nb<32>(p, wmap, xmap, s, pdl);
    case 48: return launch_nb<48>(p, wmap, xmap, s, pdl);
    case 64: return launch_nb<64>(p, wmap, xmap, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t tc_configure() {
  const int smem = 200 * 1024;
  cudaError_t e = cudaFuncSetAttribute(tcg::tc_gemm_kernel<16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tcg::tc_gemm_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tcg::tc_gemm_kernel<48>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tcg::tc_gemm_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  return e;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

cudaError_t encode_tmap_2d(CUtensorMap* map, bool bf16, const void* base, long long rows,
                           long long cols, int box_cols, int box_rows, bool swizzle128) {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f) return cudaErrorNotSupported;
    fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  const int es = bf16 ? 2 : 4;
  if (rows < 1 || cols < 1 || rows >= (1ll << 32) || cols >= (1ll << 32) ||
      (cols * es) % 16 || box_cols < 1 || box_cols > 256 || (box_cols * es) % 16 ||
      box_rows < 1 || box_rows > 256 || (reinterpret_cast<uintptr_t>(base) & 15u))
    return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * es};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r =
      fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_bf16(CUtensorMap* map, const void* base, long long rows, long long cols,
                           int box_rows) {
  if (cols % 64) return cudaErrorInvalidValue;
  return encode_tmap_2d(map, true, base, rows, cols, 64, box_rows, true);
}

}  // namespace rqk
