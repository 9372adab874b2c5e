// Decode path (M <= 64): a bandwidth-bound split-K skinny GEMM.
//
// The pages' GEMM pipeline (the guide's diagram, "Pipeline A") streams packed
// weights with cp.async, redistributes them with ldmatrix and dequantises
// with interleaved integer/float work before the MMA.  On sm_103a this kernel
// keeps the idea and changes the machinery:
//   * one elected producer thread streams each CTA's packed codes, scales and
//     zeros into a shared-memory ring with 1-D bulk async copies
//     (cp.async.bulk), and the CTA's slice of X with 2-D TMA (128-byte
//     swizzle); consumers wait on mbarriers;
//   * because the packer already stored every 32-bit word in mma.m16n8k16
//     A-fragment order, one 16-byte shared load per lane gives four MMA
//     fragments -- no ldmatrix and no runtime swizzle;
//   * dequantisation is 9 integer/half instructions per 8 weights: LOP3
//     mask-and-OR with the 0x6400 (1024.0) pattern turns nibbles into
//     1024 + q (or 1024 + 16 q), one HSUB2/HFMA2 gives q - z exactly; the
//     fp16 scale multiplies the fp32 per-group partial sum instead of the
//     weight, so no weight is rounded;
//   * W^T is the MMA's A operand (16 output columns per fragment) and X^T its
//     B operand (8 rows of X per n8 tile), so one dequantised fragment serves
//     every 8 rows of X;
//   * the K range is split over the CTAs of a thread-block cluster and the
//     partial tiles are summed through distributed shared memory in a fixed
//     rank order (deterministic, no global scratch, one launch).
#include <algorithm>

#include "tm_common.cuh"

namespace w4 {

static __device__ uint32_t s_err_decode;

struct DecodeParams {
  const uint8_t* codes;
  const uint8_t* scales;
  const uint8_t* zeros;
  __half* Y;
  int M, N, NT, KT, G;
  int nsg_total;   // pairs of groups
  int sg_per_cta;  // pairs of groups per CTA of a cluster
  int stages;
  uint32_t stage_bytes;
  uint32_t p_off;    // offset of the partial tile
  uint32_t bar_off;  // offset of the barriers
};

template <int MT, int WN, int NW, int UPS>
struct DecodeShape {
  static constexpr int CN = NW * WN;         // n-tiles per CTA
  static constexpr int CNN = CN * 16;        // columns per CTA
  static constexpr int PS = CNN + 4;         // padded row of the partial tile (floats)
  static constexpr uint32_t X_BYTES = UPS * MT * 1024;
  static constexpr uint32_t C_BYTES = CN * UPS * kUnitBytes;
  static constexpr uint32_t S_BYTES = CN * 64;
  static constexpr uint32_t Z_BYTES = CN * 16;
  static constexpr uint32_t STAGE_RAW = X_BYTES + C_BYTES + S_BYTES + Z_BYTES;
  static constexpr uint32_t STAGE = (STAGE_RAW + 1023) & ~1023u;
  static constexpr uint32_t P_BYTES = MT * 8 * PS * 4;
};

__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity) {
  unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) {
      atomicOr(&s_err_decode, kErrTimeout);
      return false;
    }
  }
  return true;
}

template <int MT, int WN, int NW, int UPS>
__global__ void __launch_bounds__((NW + 1) * 32, 2) decode_kernel(const __grid_constant__ CUtensorMap tmX,
                                                               const DecodeParams P) {
  using SH = DecodeShape<MT, WN, NW, UPS>;
  constexpr int CN = SH::CN;
  constexpr int UPG = UPS / 2;  // units (of 64 k) per group
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_base);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt0 = blockIdx.x * CN;
  const int S = gridDim.y;
  const int sg_begin = blockIdx.y * P.sg_per_cta;
  const int sg_end = min(P.nsg_total, sg_begin + P.sg_per_cta);
  const int nsg = max(0, sg_end - sg_begin);
  const int stages = P.stages;

  const uint32_t bar_full = base + P.bar_off;
  const uint32_t bar_empty = bar_full + 8 * stages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P.bar_off + 16 * stages);
  float* part = reinterpret_cast<float*>(smem + P.p_off);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, NW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == NW) {
    // ---------------- producer: one elected thread ----------------
    if (lane == 0) {
      prefetch_tmap(&tmX);
      int nvalid = min(CN, P.NT - nt0);
      if (nvalid < 0) nvalid = 0;
      const uint32_t tx = SH::X_BYTES + (uint32_t)nvalid * (UPS * kUnitBytes + 64 + 16);
      int issued = 0;
      for (int i = 0; i < nsg; ++i) {
        const int slot = i % stages;
        const uint32_t ph = (uint32_t)(i / stages) & 1u;
        if (!mbar_wait(bar_empty + 8 * slot, ph ^ 1u, abort_flag, &s_err_decode)) break;
        const int sg = sg_begin + i;
        const uint32_t full = bar_full + 8 * slot;
        const uint32_t st = base + slot * P.stage_bytes;
        mbar_expect_tx(full, tx);
#pragma unroll
        for (int u = 0; u < UPS; ++u) tma_load_2d(st + u * MT * 1024, &tmX, (sg * UPS + u) * kUnitK, 0, full);
        const uint32_t c_dst = st + SH::X_BYTES;
        const uint32_t s_dst = c_dst + SH::C_BYTES;
        const uint32_t z_dst = s_dst + SH::S_BYTES;
        for (int j = 0; j < nvalid; ++j) {
          const int nt = nt0 + j;
          bulk_g2s(c_dst + j * UPS * kUnitBytes, P.codes + ((size_t)nt * P.KT + (size_t)sg * UPS) * kUnitBytes,
                   UPS * kUnitBytes, full);
          bulk_g2s(s_dst + j * 64, P.scales + ((size_t)nt * P.G + 2 * (size_t)sg) * 32, 64, full);
          bulk_g2s(z_dst + j * 16, P.zeros + ((size_t)nt * (P.G / 2) + sg) * 16, 16, full);
        }
        ++issued;
      }
      // Never leave with copies in flight into this CTA's shared memory.
      for (int i = max(0, issued - stages); i < issued; ++i)
        drain_wait(bar_full + 8 * (i % stages), (uint32_t)(i / stages) & 1u);
    }
    __syncwarp();
  } else {
    // ---------------- consumers: NW warps, WN n-tiles each ----------------
    const int gr = lane >> 2, t = lane & 3;
    float acc[WN][MT][4];
#pragma unroll
    for (int j = 0; j < WN; ++j)
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][m][e] = 0.f;

    for (int i = 0; i < nsg; ++i) {
      const int slot = i % stages;
      const uint32_t ph = (uint32_t)(i / stages) & 1u;
      if (!mbar_wait(bar_full + 8 * slot, ph, abort_flag, &s_err_decode)) break;
      const uint32_t st = base + slot * P.stage_bytes;
      const uint32_t c_base = st + SH::X_BYTES;
      const uint32_t s_base = c_base + SH::C_BYTES;
      const uint32_t z_base = s_base + SH::S_BYTES;
#pragma unroll
      for (int gi = 0; gi < 2; ++gi) {
        float s_lo[WN], s_hi[WN];
        uint32_t zz[WN], zf[WN];
#pragma unroll
        for (int j = 0; j < WN; ++j) {
          const int jj = warp * WN + j;
          const uint32_t sp = lds32(s_base + jj * 64 + gi * 32 + gr * 4);
          s_lo[j] = __half2float(__ushort_as_half((unsigned short)(sp & 0xFFFFu)));
          s_hi[j] = __half2float(__ushort_as_half((unsigned short)(sp >> 16)));
          const uint32_t zw = lds32(z_base + jj * 16 + gi * 8 + (gr & ~3));
          const uint32_t zb = (zw >> (8 * (gr & 3))) & 0xFFu;
          zz[j] = zero_pair_lo(zb & 15u);
          zf[j] = zero_pair_hi(zb >> 4);
        }
        float tmp[WN][MT][4];
#pragma unroll
        for (int j = 0; j < WN; ++j)
#pragma unroll
          for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int e = 0; e < 4; ++e) tmp[j][m][e] = 0.f;
#pragma unroll
        for (int uu = 0; uu < UPG; ++uu) {
          const int u = gi * UPG + uu;
          // B fragments: X rows mt*8+gr, k = 16t .. 16t+15 of this unit (two
          // 16-byte chunks of a 128-byte swizzled row).
          uint4 xa[MT], xb[MT];
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const uint32_t row = st + (u * MT + m) * 1024 + gr * 128;
            xa[m] = lds128(row + (((2 * t) ^ gr) << 4));
            xb[m] = lds128(row + (((2 * t + 1) ^ gr) << 4));
          }
          uint4 cw[WN];
#pragma unroll
          for (int j = 0; j < WN; ++j)
            cw[j] = lds128(c_base + ((warp * WN + j) * UPS + u) * kUnitBytes + lane * 16);
#pragma unroll
          for (int stp = 0; stp < 4; ++stp) {
#pragma unroll
            for (int j = 0; j < WN; ++j) {
              const uint32_t w = stp == 0 ? cw[j].x : stp == 1 ? cw[j].y : stp == 2 ? cw[j].z : cw[j].w;
              uint32_t a[4];
              dequant_word(w, zz[j], zf[j], a);
#pragma unroll
              for (int m = 0; m < MT; ++m) {
                const uint32_t b0 = stp == 0 ? xa[m].x : stp == 1 ? xa[m].z : stp == 2 ? xb[m].x : xb[m].z;
                const uint32_t b1 = stp == 0 ? xa[m].y : stp == 1 ? xa[m].w : stp == 2 ? xb[m].y : xb[m].w;
                mma_16816(tmp[j][m], a, b0, b1);
              }
            }
          }
        }
#pragma unroll
        for (int j = 0; j < WN; ++j)
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            acc[j][m][0] = fmaf(s_lo[j], tmp[j][m][0], acc[j][m][0]);
            acc[j][m][1] = fmaf(s_lo[j], tmp[j][m][1], acc[j][m][1]);
            acc[j][m][2] = fmaf(s_hi[j], tmp[j][m][2], acc[j][m][2]);
            acc[j][m][3] = fmaf(s_hi[j], tmp[j][m][3], acc[j][m][3]);
          }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
    }
    // Partial tile, [m][n_local] with a padded row.
#pragma unroll
    for (int j = 0; j < WN; ++j) {
      const int nl = (warp * WN + j) * 16 + gr;
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const int r0 = m * 8 + 2 * t;
        part[r0 * SH::PS + nl] = acc[j][m][0];
        part[(r0 + 1) * SH::PS + nl] = acc[j][m][1];
        part[r0 * SH::PS + nl + 8] = acc[j][m][2];
        part[(r0 + 1) * SH::PS + nl + 8] = acc[j][m][3];
      }
    }
  }

  // ---------------- reduction over the cluster's K slices ----------------
  if (S > 1) {
    cluster_sync_all();
  } else {
    __syncthreads();
  }
  const uint32_t rank = S > 1 ? cluster_ctarank() : 0u;
  const int span = SH::CNN / S;
  const int lo = (int)rank * span;
  const int half_span = span >> 1;
  const int items = P.M * half_span;
  const uint32_t part_s = smem_u32(part);
  for (int it = threadIdx.x; it < items; it += blockDim.x) {
    const int m = it / half_span;
    const int nl = lo + 2 * (it - m * half_span);
    const int n = nt0 * 16 + nl;
    if (n >= P.N) continue;
    const uint32_t off = (uint32_t)(m * SH::PS + nl) * 4u;
    float2 v = make_float2(0.f, 0.f);
    if (S > 1) {
      for (int r = 0; r < S; ++r) {
        const float2 x = ld_dsmem_f2(map_shared_rank(part_s + off, (uint32_t)r));
        v.x += x.x;
        v.y += x.y;
      }
    } else {
      v = *reinterpret_cast<const float2*>(part + m * SH::PS + nl);
    }
    *reinterpret_cast<__half2*>(P.Y + (size_t)m * P.N + n) = __floats2half2_rn(v.x, v.y);
  }
  if (S > 1) cluster_sync_all();
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------

cudaError_t decode_error_bits(uint32_t* bits, bool clear) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, s_err_decode, sizeof(v));
  if (e != cudaSuccess) return e;
  if (clear && v) {
    uint32_t zero = 0;
    e = cudaMemcpyToSymbol(s_err_decode, &zero, sizeof(zero));
  }
  *bits = v;
  return e;
}

namespace {

constexpr int kNW = 4;
constexpr uint32_t kSmemBudget = 113 * 1024;  // two CTAs per SM

int mt_for(int M) { return M <= 8 ? 1 : M <= 16 ? 2 : M <= 32 ? 4 : 8; }

template <int MT, int WN, int UPS>
uint32_t stage_bytes() {
  return DecodeShape<MT, WN, kNW, UPS>::STAGE;
}

uint32_t stage_bytes_rt(int MT, int WN, int UPS) {
  const uint32_t CN = kNW * WN;
  const uint32_t raw = UPS * MT * 1024 + CN * UPS * kUnitBytes + CN * 64 + CN * 16;
  return (raw + 1023) & ~1023u;
}

uint32_t part_bytes_rt(int MT, int WN) { return MT * 8 * (kNW * WN * 16 + 4) * 4; }

bool valid_combo(int MT, int WN) {
  if (WN != 1 && WN != 2 && WN != 4) return false;
  return MT * WN <= 8;
}

template <int MT, int WN, int UPS>
tm_status launch_t(const CUtensorMap& tmX, const DecodeParams& P, int S, uint32_t smem, cudaStream_t stream) {
  auto kern = decode_kernel<MT, WN, kNW, UPS>;
  static bool attr_done = false;  // per instantiation, per process
  if (!attr_done) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess)
      return TM_ERR_CUDA;
    attr_done = true;
  }
  const int CN = kNW * WN;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((P.NT + CN - 1) / CN), (unsigned)S, 1);
  cfg.blockDim = dim3((kNW + 1) * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 1;
  at[0].val.clusterDim.y = (unsigned)S;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = S > 1 ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmX, P);
  return e == cudaSuccess ? TM_OK : TM_ERR_CUDA;
}

template <int MT, int WN>
tm_status launch_mw(int UPS, const CUtensorMap& tmX, const DecodeParams& P, int S, uint32_t smem,
                    cudaStream_t stream) {
  return UPS == 4 ? launch_t<MT, WN, 4>(tmX, P, S, smem, stream) : launch_t<MT, WN, 2>(tmX, P, S, smem, stream);
}

}  // namespace

tm_status plan_decode(const tm_packed* p, int M, const tm_gemm_config* in, tm_gemm_config* out) {
  const Layout& L = p->L;
  const int MT = mt_for(M);
  int tile_n = in && in->tile_n ? in->tile_n : (MT >= 8 ? 64 : 128);
  if (tile_n != 64 && tile_n != 128 && tile_n != 256) return TM_ERR_INVALID_ARG;
  const int WN = tile_n / 16 / kNW;
  if (!valid_combo(MT, WN)) return TM_ERR_UNSUPPORTED;
  const int CN = kNW * WN;
  const int NB = (L.NT + CN - 1) / CN;
  const int nsg_total = L.G / 2;
  int S = in && in->split_k ? in->split_k : 0;
  if (S == 0) {
    const int target = 2 * num_sms(p->device);
    S = 1;
    while (S < 8 && NB * S < target && 2 * S <= nsg_total) S *= 2;
  }
  if (S != 1 && S != 2 && S != 4 && S != 8) return TM_ERR_INVALID_ARG;
  const int UPS = 2 * L.g / kUnitK;
  const uint32_t sb = stage_bytes_rt(MT, WN, UPS);
  const int per_cta = (nsg_total + S - 1) / S;
  int stages = in && in->stages ? in->stages : 0;
  if (stages == 0) {
    const uint32_t fixed = part_bytes_rt(MT, WN) + 1024 + 256;
    stages = (int)((kSmemBudget - fixed) / sb);
    stages = std::max(2, std::min(stages, 6));
    stages = std::min(stages, std::max(2, per_cta));
  }
  if (stages < 2 || stages > 8) return TM_ERR_INVALID_ARG;
  out->path = 1;
  out->split_k = S;
  out->tile_n = tile_n;
  out->stages = stages;
  return TM_OK;
}

tm_status launch_decode(const void* X, const tm_packed* p, void* Y, int M, const tm_gemm_config& c,
                        cudaStream_t stream) {
  const Layout& L = p->L;
  const int MT = mt_for(M);
  const int WN = c.tile_n / 16 / kNW;
  const int S = c.split_k;
  const int UPS = 2 * L.g / kUnitK;
  // X as a 2-D tensor {K, M}: box = 64 k x (8 MT) rows, 128-byte swizzle;
  // rows beyond M and columns beyond K read as zeros.
  CUtensorMap tmX;
  {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return TM_ERR_CUDA;
    cuuint64_t dims[2] = {(cuuint64_t)L.K, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)L.K * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)(8 * MT)};
    cuuint32_t es[2] = {1, 1};
    if (fn(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(X), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return TM_ERR_CUDA;
  }
  DecodeParams P;
  P.codes = p->base + L.codes_off;
  P.scales = p->base + L.scales_off;
  P.zeros = p->base + L.zeros_off;
  P.Y = reinterpret_cast<__half*>(Y);
  P.M = M;
  P.N = L.N;
  P.NT = L.NT;
  P.KT = L.KT;
  P.G = L.G;
  P.nsg_total = L.G / 2;
  P.sg_per_cta = (P.nsg_total + S - 1) / S;
  P.stages = c.stages;
  P.stage_bytes = stage_bytes_rt(MT, WN, UPS);
  P.p_off = P.stage_bytes * c.stages;
  P.bar_off = (P.p_off + part_bytes_rt(MT, WN) + 15) & ~15u;
  const uint32_t smem = P.bar_off + 16 * c.stages + 16 + 1024;  // + alignment slack
  if (smem > 227 * 1024) return TM_ERR_UNSUPPORTED;
  tm_status st;
  switch (MT * 16 + WN) {
    case 1 * 16 + 1: st = launch_mw<1, 1>(UPS, tmX, P, S, smem, stream); break;
    case 1 * 16 + 2: st = launch_mw<1, 2>(UPS, tmX, P, S, smem, stream); break;
    case 1 * 16 + 4: st = launch_mw<1, 4>(UPS, tmX, P, S, smem, stream); break;
    case 2 * 16 + 1: st = launch_mw<2, 1>(UPS, tmX, P, S, smem, stream); break;
    case 2 * 16 + 2: st = launch_mw<2, 2>(UPS, tmX, P, S, smem, stream); break;
    case 2 * 16 + 4: st = launch_mw<2, 4>(UPS, tmX, P, S, smem, stream); break;
    case 4 * 16 + 1: st = launch_mw<4, 1>(UPS, tmX, P, S, smem, stream); break;
    case 4 * 16 + 2: st = launch_mw<4, 2>(UPS, tmX, P, S, smem, stream); break;
    case 8 * 16 + 1: st = launch_mw<8, 1>(UPS, tmX, P, S, smem, stream); break;
    default: return TM_ERR_UNSUPPORTED;
  }
  if (st == TM_OK) set_launch_count(1);
  return st;
}

}  // namespace w4
