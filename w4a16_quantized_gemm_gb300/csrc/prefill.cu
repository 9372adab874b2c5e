// Prefill path (large M): a compute-bound tensor-core GEMM on tcgen05.
//
// The pages' pipeline (the guide's diagram, "Pipeline A": asynchronous load,
// conflict-free shared memory, ILP dequantisation, tensor-core MMA) maps onto
// Blackwell's warp-specialised form:
//   * warp 0, one thread: TMA loads per 64-k block into ring A -- the X tile
//     (128 x 64 fp16, 128-byte swizzle), the packed code tile (16 n-tiles x one
//     512-byte unit), and the matching scales and zeros;
//   * warps 2..9 (256 threads): dequantise the codes in registers
//     ((q - z) exact in fp16, one fp16 multiply by s) and store the
//     BN x 64 fp16 tile W^T into ring B in the same 128-byte swizzled,
//     K-major layout TMA would write, then release it to the tensor core
//     with a proxy fence and an mbarrier arrive;
//   * warp 1, one thread: tcgen05.mma kind::f16, M = 128, N = BN, K = 16,
//     fp32 accumulators in tensor memory (TMEM); tcgen05.commit frees the
//     ring A and ring B slots it read;
//   * warps 4..7: epilogue, TMEM -> registers (tcgen05.ld) -> fp16 -> Y.
// Ring A (24.75 KB per 64-k block) is deep and ring B (32 KB) shallow, so the
// copies run far ahead of the tensor core without spending shared memory on
// dequantised tiles that wait.  Small problems split K over a cluster of S
// CTAs: after the main loop every CTA stores its fp32 tile, slice by slice,
// into the shared memory of the CTA that owns the slice (reusing ring
// memory), and each owner sums the S partials in rank order.
// All waits are bounded; a timeout raises a device error bit and the CTA
// unwinds without leaving copies or MMAs in flight.
#include <algorithm>

#include "tm_common.cuh"

namespace w4 {

static __device__ uint32_t s_err_prefill;

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kPrefillThreads = 320;  // 10 warps
constexpr int kDequantWarp0 = 2;
constexpr int kDequantWarps = 8;

template <int BN, int SA, int SB>
struct PrefillShape {
  static constexpr int NTB = BN / 16;                       // n-tiles per CTA
  // ring A slot: X tile, packed codes, scales (one group), zeros (a pair of groups)
  static constexpr uint32_t X_BYTES = kBM * kBK * 2;
  static constexpr uint32_t C_BYTES = NTB * kUnitBytes;
  static constexpr uint32_t S_BYTES = NTB * 32;
  static constexpr uint32_t Z_BYTES = NTB * 16;
  static constexpr uint32_t X_OFF = 0;
  static constexpr uint32_t C_OFF = X_BYTES;
  static constexpr uint32_t S_OFF = C_OFF + C_BYTES;
  static constexpr uint32_t Z_OFF = S_OFF + S_BYTES;
  static constexpr uint32_t A_SLOT = (Z_OFF + Z_BYTES + 1023) & ~1023u;
  static constexpr uint32_t A_TX = X_BYTES + C_BYTES + S_BYTES + Z_BYTES;
  // ring B slot: dequantised W^T tile
  static constexpr uint32_t B_SLOT = BN * kBK * 2;
  static constexpr uint32_t B_BASE = SA * A_SLOT;
  static constexpr uint32_t BAR_OFF = B_BASE + SB * B_SLOT;
  static constexpr uint32_t SMEM = BAR_OFF + 16 * (SA + SB) + 64 + 1024;  // + alignment slack
  static constexpr uint32_t RED_BYTES = kBM * BN * 4;  // split-K receive buffer (reuses the rings)
  static_assert(RED_BYTES <= BAR_OFF, "reduction buffer must fit in the rings");
};

struct PrefillParams {
  __half* Y;
  int M, N, NT, KT, G, g, UPS;
  int kb_total;   // 64-k blocks
  int kb_per_cta; // 64-k blocks per CTA of a cluster
};

__device__ __forceinline__ bool wait_time_only(uint32_t bar, uint32_t parity) {
  unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) {
      atomicOr(&s_err_prefill, kErrTimeout);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ uint32_t f2h2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int BN, int SA, int SB>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmC,
                   const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmZ,
                   const PrefillParams P) {
  using SH = PrefillShape<BN, SA, SB>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_base);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt0 = blockIdx.x * SH::NTB;
  const int m0 = blockIdx.y * kBM;
  const int S = gridDim.z;
  const int kb0 = blockIdx.z * P.kb_per_cta;
  const int nkb = max(0, min(P.kb_total, kb0 + P.kb_per_cta) - kb0);

  const uint32_t barA = base + SH::BAR_OFF;      // [SA] full, then [SA] empty
  const uint32_t barB = barA + 16 * SA;          // [SB] full, then [SB] empty
  const uint32_t bar_acc = barB + 16 * SB;       // accumulator complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SH::BAR_OFF + 16 * (SA + SB) + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SH::BAR_OFF + 16 * (SA + SB) + 12);
  auto fullA = [&](int s) { return barA + 8 * s; };
  auto emptyA = [&](int s) { return barA + 8 * (SA + s); };
  auto fullB = [&](int s) { return barB + 8 * s; };
  auto emptyB = [&](int s) { return barB + 8 * (SB + s); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < SA; ++s) {
      mbar_init(fullA(s), 1);
      mbar_init(emptyA(s), 1);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(fullB(s), kDequantWarps);
      mbar_init(emptyB(s), 1);
    }
    mbar_init(bar_acc, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_d = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer (ring A) ----------------
    if (lane == 0) {
      prefetch_tmap(&tmX);
      prefetch_tmap(&tmC);
      prefetch_tmap(&tmS);
      prefetch_tmap(&tmZ);
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int kb = kb0 + i;
        const int s = i % SA;
        const uint32_t ph = (uint32_t)(i / SA) & 1u;
        if (!mbar_wait(emptyA(s), ph ^ 1u, abort_flag, &s_err_prefill)) break;
        const uint32_t st = base + s * SH::A_SLOT;
        const int grp = kb * kBK / P.g;
        mbar_expect_tx(fullA(s), SH::A_TX);
        tma_load_2d(st + SH::X_OFF, &tmX, kb * kBK, m0, fullA(s));
        tma_load_4d(st + SH::C_OFF, &tmC, 0, kb % P.UPS, nt0, kb / P.UPS, fullA(s));
        tma_load_4d(st + SH::S_OFF, &tmS, 0, grp & 1, nt0, grp >> 1, fullA(s));
        tma_load_3d(st + SH::Z_OFF, &tmZ, 0, nt0, grp >> 1, fullA(s));
        ++issued;
      }
      for (int i = max(0, issued - SA); i < issued; ++i)
        wait_time_only(fullA(i % SA), (uint32_t)(i / SA) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(kBM, BN);
      for (int i = 0; i < nkb; ++i) {
        const int sa = i % SA, sb = i % SB;
        const uint32_t pa = (uint32_t)(i / SA) & 1u, pb = (uint32_t)(i / SB) & 1u;
        if (!mbar_wait(fullA(sa), pa, abort_flag, &s_err_prefill)) break;
        if (!mbar_wait(fullB(sb), pb, abort_flag, &s_err_prefill)) break;
        tc_fence_after();
        const uint64_t da = smem_desc_sw128(base + sa * SH::A_SLOT + SH::X_OFF);
        const uint64_t db = smem_desc_sw128(base + SH::B_BASE + sb * SH::B_SLOT);
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          // advance 16 fp16 (32 bytes) along K inside the swizzle atom
          tc_mma_f16(tmem_d, da + (uint64_t)(2 * k), db + (uint64_t)(2 * k), idesc, (i > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit(emptyA(sa));
        tc_commit(emptyB(sb));
      }
      // Completes once every MMA issued above has finished (also on abort).
      tc_commit(bar_acc);
    }
    __syncwarp();
  } else {
    // ---------------- dequantisers (warps 2..9) ----------------
    const int d = threadIdx.x - kDequantWarp0 * 32;  // 0..255
    constexpr int SLOTS = SH::NTB * 32;               // lane-slots per k-block
    constexpr int PER = SLOTS / (kDequantWarps * 32);
    for (int i = 0; i < nkb; ++i) {
      const int kb = kb0 + i;
      const int sa = i % SA, sb = i % SB;
      const uint32_t pa = (uint32_t)(i / SA) & 1u, pb = (uint32_t)(i / SB) & 1u;
      if (!mbar_wait(fullA(sa), pa, abort_flag, &s_err_prefill)) break;
      if (!mbar_wait(emptyB(sb), pb ^ 1u, abort_flag, &s_err_prefill)) break;
      const uint32_t st = base + sa * SH::A_SLOT;
      const uint32_t bt = base + SH::B_BASE + sb * SH::B_SLOT;
      const int grp = kb * kBK / P.g;
#pragma unroll
      for (int r = 0; r < PER; ++r) {
        const int slot = d + r * kDequantWarps * 32;
        const int j = slot >> 5, ln = slot & 31;
        const int gr = ln >> 2, t = ln & 3;
        const uint4 cw = lds128(st + SH::C_OFF + j * kUnitBytes + ln * 16);
        const uint32_t sp = lds32(st + SH::S_OFF + j * 32 + gr * 4);
        const uint32_t zw = lds32(st + SH::Z_OFF + j * 16 + (grp & 1) * 8 + (gr & ~3));
        const uint32_t zb = (zw >> (8 * (gr & 3))) & 0xFFu;
        const uint32_t zz = zero_pair_lo(zb & 15u), zf = zero_pair_hi(zb >> 4);
        const uint32_t s_lo = (sp & 0xFFFFu) | (sp << 16);      // s of row gr, twice
        const uint32_t s_hi = (sp >> 16) | (sp & 0xFFFF0000u);  // s of row gr+8, twice
        uint32_t a0[4], a1[4], a2[4], a3[4];
        dequant_word(cw.x, zz, zf, a0);
        dequant_word(cw.y, zz, zf, a1);
        dequant_word(cw.z, zz, zf, a2);
        dequant_word(cw.w, zz, zf, a3);
        const int row_lo = j * 16 + gr, row_hi = row_lo + 8;
        const uint32_t b_lo = bt + row_lo * 128;
        const uint32_t b_hi = bt + row_hi * 128;
        // row gr: k 16t..16t+7 (chunk 2t) and 16t+8..16t+15 (chunk 2t+1); 128-byte swizzle
        sts128(b_lo + (((2 * t) ^ gr) << 4), hmul2_u32(a0[0], s_lo), hmul2_u32(a0[2], s_lo), hmul2_u32(a1[0], s_lo),
               hmul2_u32(a1[2], s_lo));
        sts128(b_lo + (((2 * t + 1) ^ gr) << 4), hmul2_u32(a2[0], s_lo), hmul2_u32(a2[2], s_lo),
               hmul2_u32(a3[0], s_lo), hmul2_u32(a3[2], s_lo));
        sts128(b_hi + (((2 * t) ^ gr) << 4), hmul2_u32(a0[1], s_hi), hmul2_u32(a0[3], s_hi), hmul2_u32(a1[1], s_hi),
               hmul2_u32(a1[3], s_hi));
        sts128(b_hi + (((2 * t + 1) ^ gr) << 4), hmul2_u32(a2[1], s_hi), hmul2_u32(a2[3], s_hi),
               hmul2_u32(a3[1], s_hi), hmul2_u32(a3[3], s_hi));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(fullB(sb));
    }
  }

  // ---------------- epilogue ----------------
  const bool epi = warp >= 4 && warp < 8;  // warps 4..7 own TMEM lanes 32*(warp%4)
  const int q = warp & 3;
  const int row = q * 32 + lane;           // accumulator row of this thread
  bool acc_ok = true;
  if (epi) {
    acc_ok = mbar_wait(bar_acc, 0, abort_flag, &s_err_prefill);
    tc_fence_after();
  }
  if (S == 1) {
    if (epi && acc_ok) {
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tc_ld_32x32b_x32(tmem_d + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * 32), v);
        tc_wait_ld();
        const int n = nt0 * 16 + c * 32;
        if (m0 + row < P.M) {
          __half* y = P.Y + (size_t)(m0 + row) * P.N + n;
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            if (n + h * 8 + 8 <= P.N) {
              uint4 o;
              o.x = f2h2(__uint_as_float(v[8 * h + 0]), __uint_as_float(v[8 * h + 1]));
              o.y = f2h2(__uint_as_float(v[8 * h + 2]), __uint_as_float(v[8 * h + 3]));
              o.z = f2h2(__uint_as_float(v[8 * h + 4]), __uint_as_float(v[8 * h + 5]));
              o.w = f2h2(__uint_as_float(v[8 * h + 6]), __uint_as_float(v[8 * h + 7]));
              *reinterpret_cast<uint4*>(y + h * 8) = o;
            }
          }
        }
      }
    }
  } else {
    // Split K: every CTA's rings are idle once all of the cluster passes this
    // barrier (MMAs finished, copies drained), so partial tiles may land there.
    cluster_sync_all();
    const int span = BN / S;
    const uint32_t my_rank = cluster_ctarank();
    const uint32_t red_s = base;  // red[rank][128 rows][span] fp32, over the rings
    if (epi) {
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        if (acc_ok && nkb > 0) {  // a CTA with no K blocks contributes zeros
          tc_ld_32x32b_x32(tmem_d + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * 32), v);
          tc_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        const int owner = (c * 32) / span;
        const int col0 = c * 32 - owner * span;
        const uint32_t dst =
            map_shared_rank(red_s + (uint32_t)(((int)my_rank * kBM + row) * span + col0) * 4u, (uint32_t)owner);
#pragma unroll
        for (int e = 0; e < 32; e += 4) st_dsmem_v4(dst + e * 4, v[e], v[e + 1], v[e + 2], v[e + 3]);
      }
    }
    cluster_sync_all();
    const float* red = reinterpret_cast<const float*>(smem);
    const int half_span = span >> 1;
    const int items = kBM * half_span;
    const int n_base = nt0 * 16 + (int)my_rank * span;
    for (int it = threadIdx.x; it < items; it += blockDim.x) {
      const int r = it / half_span;
      const int col = 2 * (it - r * half_span);
      const int n = n_base + col;
      if (m0 + r >= P.M || n >= P.N) continue;
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll 8
      for (int k = 0; k < S; ++k) {
        const float2 x = *reinterpret_cast<const float2*>(red + (k * kBM + r) * span + col);
        acc.x += x.x;
        acc.y += x.y;
      }
      *reinterpret_cast<uint32_t*>(P.Y + (size_t)(m0 + r) * P.N + n) = f2h2(acc.x, acc.y);
    }
  }
  if (warp == 1 && lane == 0) {
    // No MMA may still run when TMEM is released.
    wait_time_only(bar_acc, 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_d, BN);
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------

cudaError_t prefill_error_bits(uint32_t* bits, bool clear) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, s_err_prefill, sizeof(v));
  if (e != cudaSuccess) return e;
  if (clear && v) {
    uint32_t zero = 0;
    e = cudaMemcpyToSymbol(s_err_prefill, &zero, sizeof(zero));
  }
  *bits = v;
  return e;
}

namespace {

constexpr int kSA = 6;  // ring A slots (X + codes + scales + zeros)
constexpr int kSB = 2;  // ring B slots (dequantised W^T)

template <int BN, int SA, int SB>
tm_status launch_t(const CUtensorMap& tmX, const tm_packed* p, const PrefillParams& P, int S, cudaStream_t stream) {
  using SH = PrefillShape<BN, SA, SB>;
  auto kern = prefill_kernel<BN, SA, SB>;
  static std::atomic<unsigned long long> attr_done{0};  // one bit per device
  if (!smem_attr_once(attr_done, (const void*)kern, (int)SH::SMEM)) return TM_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((P.NT + SH::NTB - 1) / SH::NTB), (unsigned)((P.M + kBM - 1) / kBM), (unsigned)S);
  cfg.blockDim = dim3(kPrefillThreads, 1, 1);
  cfg.dynamicSmemBytes = SH::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 1;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = (unsigned)S;
  cfg.attrs = at;
  cfg.numAttrs = S > 1 ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmX, p->tm_codes, p->tm_scales, p->tm_zeros, P);
  return e == cudaSuccess ? TM_OK : TM_ERR_CUDA;
}

}  // namespace

// Split K only when the output tiles cannot fill the GPU: the smallest
// power of two (up to 8) that brings the CTA count to about one per SM,
// keeping at least 8 blocks of 64 k per CTA.
tm_status plan_prefill(const tm_packed* p, int M, const tm_gemm_config* in, tm_gemm_config* out) {
  const Layout& L = p->L;
  const int tile_n = in && in->tile_n ? in->tile_n : 256;
  if (tile_n != 256) return TM_ERR_UNSUPPORTED;
  const int want_S = in ? in->split_k : 0;
  if (want_S && want_S != 1 && want_S != 2 && want_S != 4 && want_S != 8) return TM_ERR_INVALID_ARG;
  if (in && in->stages && in->stages != kSA) return TM_ERR_UNSUPPORTED;
  const int tiles = ((M + kBM - 1) / kBM) * ((L.NT + 15) / 16);
  const int kb = L.Kp / kBK;
  int S = want_S;
  if (!S) {
    const int sms = num_sms(p->device);
    S = 1;
    while (S < 8 && tiles * S < (sms * 4) / 5 && kb / (2 * S) >= 8) S *= 2;
  }
  out->path = 2;
  out->split_k = S;
  out->tile_n = tile_n;
  out->stages = kSA;
  out->warp_n = 0;
  out->tile_m = 0;
  return TM_OK;
}

tm_status launch_prefill(const void* X, const tm_packed* p, void* Y, int M, const tm_gemm_config& c,
                         cudaStream_t stream) {
  const Layout& L = p->L;
  CUtensorMap tmX;
  {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return TM_ERR_CUDA;
    cuuint64_t dims[2] = {(cuuint64_t)L.K, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)L.K * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBM};
    cuuint32_t es[2] = {1, 1};
    if (fn(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(X), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return TM_ERR_CUDA;
  }
  PrefillParams P;
  P.Y = reinterpret_cast<__half*>(Y);
  P.M = M;
  P.N = L.N;
  P.NT = L.NT;
  P.KT = L.KT;
  P.G = L.G;
  P.g = L.g;
  P.UPS = L.UPS;
  P.kb_total = L.Kp / kBK;
  const int S = c.split_k;
  P.kb_per_cta = (P.kb_total + S - 1) / S;
  tm_status st = TM_ERR_UNSUPPORTED;
  if (c.tile_n == 256 && c.stages == kSA) st = launch_t<256, kSA, kSB>(tmX, p, P, S, stream);
  if (st == TM_OK) set_launch_count(1);
  return st;
}

}  // namespace w4
