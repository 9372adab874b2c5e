// Prefill path (large M): a compute-bound tensor-core GEMM on tcgen05.
//
// The pages' pipeline (the guide's diagram, "Pipeline A": asynchronous load,
// conflict-free shared memory, ILP dequantisation, tensor-core MMA) maps onto
// Blackwell's warp-specialised form:
//   * warp 0, one thread: TMA loads per 64-k block -- the X tile
//     (128 x 64 fp16, 128-byte swizzle), the packed code tile (16 n-tiles x one
//     512-byte unit), and the matching scales and zeros;
//   * warps 2..9 (256 threads): dequantise the codes in registers
//     ((q - z) exact in fp16, one fp16 multiply by s) and store the
//     BN x 64 fp16 tile W^T into shared memory in the same 128-byte swizzled,
//     K-major layout TMA would write, then release it to the tensor core
//     with a proxy fence and an mbarrier arrive;
//   * warp 1, one thread: tcgen05.mma kind::f16, M = 128, N = BN, K = 16,
//     fp32 accumulators in tensor memory (TMEM); tcgen05.commit frees each
//     stage;
//   * warps 4..7: epilogue, TMEM -> registers (tcgen05.ld) -> fp16 -> Y.
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

template <int BN>
struct PrefillShape {
  static constexpr int NTB = BN / 16;                       // n-tiles per CTA
  static constexpr uint32_t A_BYTES = kBM * kBK * 2;        // X tile
  static constexpr uint32_t B_BYTES = BN * kBK * 2;         // dequantised W^T tile
  static constexpr uint32_t C_BYTES = NTB * kUnitBytes;     // packed codes
  static constexpr uint32_t S_BYTES = NTB * 32;             // scales (one group)
  static constexpr uint32_t Z_BYTES = NTB * 16;             // zeros (a pair of groups)
  static constexpr uint32_t A_OFF = 0;
  static constexpr uint32_t B_OFF = A_BYTES;
  static constexpr uint32_t C_OFF = B_OFF + B_BYTES;
  static constexpr uint32_t S_OFF = C_OFF + C_BYTES;
  static constexpr uint32_t Z_OFF = S_OFF + S_BYTES;
  static constexpr uint32_t STAGE = (Z_OFF + Z_BYTES + 1023) & ~1023u;
  static constexpr uint32_t TX = A_BYTES + C_BYTES + S_BYTES + Z_BYTES;
};

struct PrefillParams {
  __half* Y;
  int M, N, NT, KT, G, g, UPS;
  int kb_total;  // 64-k blocks
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

template <int BN, int STAGES>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmC,
                   const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmZ,
                   const PrefillParams P) {
  using SH = PrefillShape<BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_base);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_blk = blockIdx.x, m_blk = blockIdx.y;
  const int nt0 = n_blk * SH::NTB;
  const int m0 = m_blk * kBM;
  const int nkb = P.kb_total;

  const uint32_t bar0 = base + STAGES * SH::STAGE;
  const uint32_t bar_tma = bar0;                    // [STAGES] X + codes + meta landed
  const uint32_t bar_deq = bar0 + 8 * STAGES;       // [STAGES] W^T tile written
  const uint32_t bar_empty = bar0 + 16 * STAGES;    // [STAGES] MMAs done reading the stage
  const uint32_t bar_acc = bar0 + 24 * STAGES;      // accumulator complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + STAGES * SH::STAGE + 24 * STAGES + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + STAGES * SH::STAGE + 24 * STAGES + 12);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_tma + 8 * s, 1);
      mbar_init(bar_deq + 8 * s, kDequantWarps);
      mbar_init(bar_empty + 8 * s, 1);
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
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tmap(&tmX);
      prefetch_tmap(&tmC);
      prefetch_tmap(&tmS);
      prefetch_tmap(&tmZ);
      int issued = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % STAGES;
        const uint32_t ph = (uint32_t)(kb / STAGES) & 1u;
        if (!mbar_wait(bar_empty + 8 * s, ph ^ 1u, abort_flag, &s_err_prefill)) break;
        const uint32_t st = base + s * SH::STAGE;
        const uint32_t full = bar_tma + 8 * s;
        const int grp = kb * kBK / P.g;
        mbar_expect_tx(full, SH::TX);
        tma_load_2d(st + SH::A_OFF, &tmX, kb * kBK, m0, full);
        tma_load_4d(st + SH::C_OFF, &tmC, 0, kb % P.UPS, nt0, kb / P.UPS, full);
        tma_load_4d(st + SH::S_OFF, &tmS, 0, grp & 1, nt0, grp >> 1, full);
        tma_load_3d(st + SH::Z_OFF, &tmZ, 0, nt0, grp >> 1, full);
        ++issued;
      }
      for (int i = max(0, issued - STAGES); i < issued; ++i)
        wait_time_only(bar_tma + 8 * (i % STAGES), (uint32_t)(i / STAGES) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(kBM, BN);
      int done = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % STAGES;
        const uint32_t ph = (uint32_t)(kb / STAGES) & 1u;
        if (!mbar_wait(bar_tma + 8 * s, ph, abort_flag, &s_err_prefill)) break;
        if (!mbar_wait(bar_deq + 8 * s, ph, abort_flag, &s_err_prefill)) break;
        tc_fence_after();
        const uint32_t st = base + s * SH::STAGE;
        const uint64_t da = smem_desc_sw128(st + SH::A_OFF);
        const uint64_t db = smem_desc_sw128(st + SH::B_OFF);
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          // advance 16 fp16 (32 bytes) along K inside the swizzle atom
          tc_mma_f16(tmem_d, da + (uint64_t)(2 * k), db + (uint64_t)(2 * k), idesc, (kb > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit(bar_empty + 8 * s);
        ++done;
      }
      // Completes once every MMA issued above has finished (also on abort).
      tc_commit(bar_acc);
      (void)done;
    }
    __syncwarp();
  } else if (warp >= kDequantWarp0 && warp < kDequantWarp0 + kDequantWarps) {
    // ---------------- dequantisers ----------------
    const int d = threadIdx.x - kDequantWarp0 * 32;  // 0..255
    constexpr int SLOTS = SH::NTB * 32;               // lane-slots per k-block
    constexpr int PER = SLOTS / (kDequantWarps * 32);
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (uint32_t)(kb / STAGES) & 1u;
      if (!mbar_wait(bar_tma + 8 * s, ph, abort_flag, &s_err_prefill)) break;
      const uint32_t st = base + s * SH::STAGE;
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
        const uint32_t s_lo = (sp & 0xFFFFu) | (sp << 16);   // s of row gr, twice
        const uint32_t s_hi = (sp >> 16) | (sp & 0xFFFF0000u);  // s of row gr+8, twice
        uint32_t a0[4], a1[4], a2[4], a3[4];
        dequant_word(cw.x, zz, zf, a0);
        dequant_word(cw.y, zz, zf, a1);
        dequant_word(cw.z, zz, zf, a2);
        dequant_word(cw.w, zz, zf, a3);
        const int row_lo = j * 16 + gr, row_hi = row_lo + 8;
        const uint32_t b_lo = st + SH::B_OFF + row_lo * 128;
        const uint32_t b_hi = st + SH::B_OFF + row_hi * 128;
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
      if (lane == 0) mbar_arrive(bar_deq + 8 * s);
    }
  }

  // ---------------- epilogue: warps 4..7 read TMEM lanes 32*(warp%4) ----------------
  if (warp >= 4 && warp < 8) {
    const bool ok = mbar_wait(bar_acc, 0, abort_flag, &s_err_prefill);
    tc_fence_after();
    const int q = warp & 3;
    const int row = m0 + q * 32 + lane;
    if (ok) {
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tc_ld_32x32b_x32(tmem_d + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * 32), v);
        tc_wait_ld();
        const int n = (nt0 * 16) + c * 32;
        if (row < P.M) {
          __half* y = P.Y + (size_t)row * P.N + n;
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            if (n + h * 8 + 8 <= P.N) {
              uint4 o;
              __half2 p0 = __floats2half2_rn(__uint_as_float(v[8 * h + 0]), __uint_as_float(v[8 * h + 1]));
              __half2 p1 = __floats2half2_rn(__uint_as_float(v[8 * h + 2]), __uint_as_float(v[8 * h + 3]));
              __half2 p2 = __floats2half2_rn(__uint_as_float(v[8 * h + 4]), __uint_as_float(v[8 * h + 5]));
              __half2 p3 = __floats2half2_rn(__uint_as_float(v[8 * h + 6]), __uint_as_float(v[8 * h + 7]));
              o.x = *reinterpret_cast<uint32_t*>(&p0);
              o.y = *reinterpret_cast<uint32_t*>(&p1);
              o.z = *reinterpret_cast<uint32_t*>(&p2);
              o.w = *reinterpret_cast<uint32_t*>(&p3);
              *reinterpret_cast<uint4*>(y + h * 8) = o;
            }
          }
        }
      }
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

template <int BN, int STAGES>
tm_status launch_t(const CUtensorMap& tmX, const tm_packed* p, const PrefillParams& P, cudaStream_t stream) {
  using SH = PrefillShape<BN>;
  auto kern = prefill_kernel<BN, STAGES>;
  const uint32_t smem = STAGES * SH::STAGE + 24 * STAGES + 64 + 1024;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return TM_ERR_CUDA;
    attr_done = true;
  }
  dim3 grid((unsigned)((P.NT + SH::NTB - 1) / SH::NTB), (unsigned)((P.M + kBM - 1) / kBM), 1);
  kern<<<grid, kPrefillThreads, smem, stream>>>(tmX, p->tm_codes, p->tm_scales, p->tm_zeros, P);
  return cudaGetLastError() == cudaSuccess ? TM_OK : TM_ERR_CUDA;
}

}  // namespace

tm_status plan_prefill(const tm_packed* p, int M, const tm_gemm_config* in, tm_gemm_config* out) {
  (void)p;
  (void)M;
  int tile_n = in && in->tile_n ? in->tile_n : 256;
  if (tile_n != 256) return TM_ERR_UNSUPPORTED;
  int S = in && in->split_k ? in->split_k : 1;
  if (S != 1) return TM_ERR_UNSUPPORTED;
  int stages = in && in->stages ? in->stages : 3;
  if (stages != 3) return TM_ERR_UNSUPPORTED;
  out->path = 2;
  out->split_k = S;
  out->tile_n = tile_n;
  out->stages = stages;
  out->warp_n = 0;
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
  tm_status st = TM_ERR_UNSUPPORTED;
  if (c.tile_n == 256 && c.stages == 3) st = launch_t<256, 3>(tmX, p, P, stream);
  if (st == TM_OK) set_launch_count(1);
  return st;
}

}  // namespace w4
