// Decode path (M <= 64): a bandwidth-bound split-K skinny GEMM.
//
// The pages' GEMM pipeline (the guide's diagram, "Pipeline A") streams packed
// weights with cp.async, redistributes them with ldmatrix and dequantises
// with interleaved integer/float work before the MMA.  On sm_103a this kernel
// keeps the idea and changes the machinery:
//   * one elected producer thread streams each CTA's packed codes, scales and
//     zeros into a shared-memory ring with three 1-D bulk async copies
//     (cp.async.bulk) per stage, and the CTA's slice of X with 2-D TMA
//     (128-byte swizzle); consumers wait on mbarriers;
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
//   * the K range is split over the CTAs of a thread-block cluster: every CTA
//     stores its partial tile slice by slice into the shared memory of the
//     CTA that owns the slice, one cluster barrier follows, and each CTA sums
//     its slice in a fixed rank order (deterministic, no global scratch);
//   * programmatic dependent launch: the weight stream starts before the
//     preceding kernel in the stream has finished; only the X loads and the
//     Y stores wait for it.
#include <algorithm>

#include "tm_common.cuh"

namespace w4 {

static __device__ uint32_t s_err_decode;

struct DecodeParams {
  const uint8_t* codes;
  const uint8_t* scales;
  const uint8_t* zeros;
  __half* Y;
  int M, N, NT;
  int nsg_total;   // pairs of groups
  int sg_per_cta;  // pairs of groups per CTA of a cluster
  int stages;
  uint32_t stage_bytes;
  uint32_t r_off;    // offset of the reduction buffer
  uint32_t bar_off;  // offset of the barriers
};

template <int MT, int WN, int NW, int UPS>
struct DecodeShape {
  static constexpr int CN = NW * WN;   // n-tiles per CTA
  static constexpr int CNN = CN * 16;  // columns per CTA
  static constexpr uint32_t X_BYTES = UPS * MT * 1024;
  static constexpr uint32_t C_BYTES = CN * UPS * kUnitBytes;
  static constexpr uint32_t S_BYTES = CN * 64;
  static constexpr uint32_t Z_BYTES = CN * 16;
  static constexpr uint32_t STAGE_RAW = X_BYTES + C_BYTES + S_BYTES + Z_BYTES;
  static constexpr uint32_t STAGE = (STAGE_RAW + 1023) & ~1023u;
  static constexpr uint32_t R_BYTES = MT * 8 * CNN * 4;  // [S][MT*8][span] floats
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
__global__ void __launch_bounds__((NW + 1) * 32) decode_kernel(const __grid_constant__ CUtensorMap tmX,
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
  float* red = reinterpret_cast<float*>(smem + P.r_off);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, NW);
    }
    *abort_flag = 0;
    fence_mbar_init();
    launch_dependents();
  }
  __syncthreads();
  // Every CTA of the cluster must be running before any CTA stores into its
  // shared memory: arrive now, wait right before the first remote store.
  if (S > 1) cluster_arrive_relaxed();

  if (warp == NW) {
    // ---------------- producer: one elected thread ----------------
    if (lane == 0) {
      prefetch_tmap(&tmX);
      const int nvalid = min(CN, P.NT - nt0);
      const uint32_t tx = SH::X_BYTES + (uint32_t)nvalid * (UPS * kUnitBytes + 64 + 16);
      auto issue_weights = [&](int i) {
        const int slot = i % stages;
        const int sg = sg_begin + i;
        const uint32_t full = bar_full + 8 * slot;
        const uint32_t c_dst = base + slot * P.stage_bytes + SH::X_BYTES;
        const uint32_t s_dst = c_dst + SH::C_BYTES;
        const uint32_t z_dst = s_dst + SH::S_BYTES;
        // one contiguous run each: codes, scales and zeros of n-tiles nt0.. for super-group sg
        const size_t row = (size_t)sg * P.NT + nt0;
        bulk_g2s(c_dst, P.codes + row * (UPS * kUnitBytes), (uint32_t)nvalid * UPS * kUnitBytes, full);
        bulk_g2s(s_dst, P.scales + row * 64, (uint32_t)nvalid * 64, full);
        bulk_g2s(z_dst, P.zeros + row * 16, (uint32_t)nvalid * 16, full);
      };
      auto issue_x = [&](int i) {
        const int slot = i % stages;
        const int sg = sg_begin + i;
        const uint32_t st = base + slot * P.stage_bytes;
#pragma unroll
        for (int u = 0; u < UPS; ++u)
          tma_load_2d(st + u * MT * 1024, &tmX, (sg * UPS + u) * kUnitK, 0, bar_full + 8 * slot);
      };
      // Fill the ring with weights first: they do not depend on the
      // preceding kernel.  X does, so its loads wait for that grid.
      const int first = min(nsg, stages);
      for (int i = 0; i < first; ++i) {
        mbar_expect_tx(bar_full + 8 * (i % stages), tx);
        issue_weights(i);
      }
      grid_dependency_wait();
      for (int i = 0; i < first; ++i) issue_x(i);
      int issued = first;
      int slot = first % stages;
      uint32_t ph = (uint32_t)(first / stages) & 1u;
      for (int i = first; i < nsg; ++i) {
        if (!mbar_wait(bar_empty + 8 * slot, ph ^ 1u, abort_flag, &s_err_decode)) break;
        mbar_expect_tx(bar_full + 8 * slot, tx);
        issue_weights(i);
        issue_x(i);
        ++issued;
        if (++slot == stages) {
          slot = 0;
          ph ^= 1u;
        }
      }
      // Never leave with copies in flight into this CTA's shared memory.
      for (int i = max(0, issued - stages); i < issued; ++i)
        drain_wait(bar_full + 8 * (i % stages), (uint32_t)(i / stages) & 1u);
    }
    __syncwarp();
    if (S > 1) cluster_wait();
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

    int slot = 0;
    uint32_t ph = 0;
    for (int i = 0; i < nsg; ++i) {
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
          // 16-byte chunks of a 128-byte swizzled row).  Rows at or past M
          // are zeros in shared memory; they are not loaded at all.
          uint4 xa[MT], xb[MT];
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            if (m * 8 + gr < P.M) {
              const uint32_t row = st + (u * MT + m) * 1024 + gr * 128;
              xa[m] = lds128(row + (((2 * t) ^ gr) << 4));
              xb[m] = lds128(row + (((2 * t + 1) ^ gr) << 4));
            } else {
              xa[m] = make_uint4(0, 0, 0, 0);
              xb[m] = make_uint4(0, 0, 0, 0);
            }
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
      if (++slot == stages) {
        slot = 0;
        ph ^= 1u;
      }
    }

    // Partial tile -> the owner of each column slice: red[rank][m][col] in
    // the owner's shared memory (its own when S == 1).
    const int span = SH::CNN / S;
    const uint32_t my_rank = S > 1 ? cluster_ctarank() : 0u;
    const uint32_t red_s = smem_u32(red);
    if (S > 1) cluster_wait();
#pragma unroll
    for (int j = 0; j < WN; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int nl = (warp * WN + j) * 16 + gr + ((e & 2) ? 8 : 0);
        const int owner = nl / span;
        const int col = nl - owner * span;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const int mm = m * 8 + 2 * t + (e & 1);
          const uint32_t off = (uint32_t)(((int)my_rank * (MT * 8) + mm) * span + col) * 4u;
          if (S > 1) {
            st_dsmem_f32(map_shared_rank(red_s + off, (uint32_t)owner), acc[j][m][e]);
          } else {
            red[off / 4] = acc[j][m][e];
          }
        }
      }
    }
  }

  // ---------------- reduction of this CTA's column slice ----------------
  if (S > 1) {
    cluster_sync_all();
  } else {
    __syncthreads();
  }
  grid_dependency_wait();  // Y may still be read by the preceding grid
  const int span = SH::CNN / S;
  const uint32_t my_rank = S > 1 ? cluster_ctarank() : 0u;
  const int half_span = span >> 1;
  const int items = P.M * half_span;
  const int n_base = nt0 * 16 + (int)my_rank * span;
  for (int it = threadIdx.x; it < items; it += blockDim.x) {
    const int m = it / half_span;
    const int col = 2 * (it - m * half_span);
    const int n = n_base + col;
    if (n >= P.N) continue;
    float2 v = make_float2(0.f, 0.f);
#pragma unroll 8
    for (int r = 0; r < S; ++r) {
      const float2 x = *reinterpret_cast<const float2*>(red + (r * (MT * 8) + m) * span + col);
      v.x += x.x;
      v.y += x.y;
    }
    *reinterpret_cast<__half2*>(P.Y + (size_t)m * P.N + n) = __floats2half2_rn(v.x, v.y);
  }
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

constexpr uint32_t kSmemBudget = 113 * 1024;  // two CTAs per SM at least

int mt_for(int M) { return M <= 8 ? 1 : M <= 16 ? 2 : M <= 32 ? 4 : 8; }

// tile_n -> (WN, NW)
bool tile_shape(int tile_n, int MT, int* WN, int* NW) {
  switch (tile_n) {
    case 64: *WN = 1; *NW = 4; return true;
    case 128: *WN = 1; *NW = 8; return true;
    case 256: *WN = 2; *NW = 8; return MT <= 4;
  }
  return false;
}

uint32_t stage_bytes_rt(int MT, int CN, int UPS) {
  const uint32_t raw = UPS * MT * 1024 + CN * UPS * kUnitBytes + CN * 64 + CN * 16;
  return (raw + 1023) & ~1023u;
}

uint32_t red_bytes_rt(int MT, int CN) { return MT * 8 * CN * 16 * 4; }

template <int MT, int WN, int NW, int UPS>
tm_status launch_t(const CUtensorMap& tmX, const DecodeParams& P, int S, uint32_t smem, cudaStream_t stream) {
  auto kern = decode_kernel<MT, WN, NW, UPS>;
  static bool attr_done = false;  // per instantiation, per process
  if (!attr_done) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess)
      return TM_ERR_CUDA;
    attr_done = true;
  }
  constexpr int CN = NW * WN;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((P.NT + CN - 1) / CN), (unsigned)S, 1);
  cfg.blockDim = dim3((NW + 1) * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  int na = 0;
  at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (S > 1) {
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = 1;
    at[na].val.clusterDim.y = (unsigned)S;
    at[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmX, P);
  return e == cudaSuccess ? TM_OK : TM_ERR_CUDA;
}

template <int MT, int WN, int NW>
tm_status launch_u(int UPS, const CUtensorMap& tmX, const DecodeParams& P, int S, uint32_t smem,
                   cudaStream_t stream) {
  return UPS == 4 ? launch_t<MT, WN, NW, 4>(tmX, P, S, smem, stream)
                  : launch_t<MT, WN, NW, 2>(tmX, P, S, smem, stream);
}

template <int MT>
tm_status launch_m(int tile_n, int UPS, const CUtensorMap& tmX, const DecodeParams& P, int S, uint32_t smem,
                   cudaStream_t stream) {
  if (tile_n == 64) return launch_u<MT, 1, 4>(UPS, tmX, P, S, smem, stream);
  if (tile_n == 128) return launch_u<MT, 1, 8>(UPS, tmX, P, S, smem, stream);
  if constexpr (MT <= 4) {
    if (tile_n == 256) return launch_u<MT, 2, 8>(UPS, tmX, P, S, smem, stream);
  }
  return TM_ERR_UNSUPPORTED;
}

}  // namespace

tm_status plan_decode(const tm_packed* p, int M, const tm_gemm_config* in, tm_gemm_config* out) {
  const Layout& L = p->L;
  const int MT = mt_for(M);
  int tile_n = in && in->tile_n ? in->tile_n : 128;
  int WN = 0, NW = 0;
  if (tile_n != 64 && tile_n != 128 && tile_n != 256) return TM_ERR_INVALID_ARG;
  if (!tile_shape(tile_n, MT, &WN, &NW)) return TM_ERR_UNSUPPORTED;
  const int CN = NW * WN;
  const int NB = (L.NT + CN - 1) / CN;
  int S = in && in->split_k ? in->split_k : 0;
  if (S == 0) {
    const int target = 2 * num_sms(p->device);
    S = 1;
    while (S < 8 && NB * S < target && 2 * S <= L.NSG) S *= 2;
  }
  if (S != 1 && S != 2 && S != 4 && S != 8) return TM_ERR_INVALID_ARG;
  const uint32_t sb = stage_bytes_rt(MT, CN, L.UPS);
  const int per_cta = (L.NSG + S - 1) / S;
  int stages = in && in->stages ? in->stages : 0;
  if (stages == 0) {
    const uint32_t fixed = red_bytes_rt(MT, CN) + 1024 + 256;
    stages = (int)((kSmemBudget - fixed) / sb);
    stages = std::max(2, std::min(stages, 4));
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
  int WN = 0, NW = 0;
  if (!tile_shape(c.tile_n, MT, &WN, &NW)) return TM_ERR_UNSUPPORTED;
  const int CN = WN * NW;
  const int S = c.split_k;
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
  P.nsg_total = L.NSG;
  P.sg_per_cta = (P.nsg_total + S - 1) / S;
  P.stages = c.stages;
  P.stage_bytes = stage_bytes_rt(MT, CN, L.UPS);
  P.r_off = P.stage_bytes * c.stages;
  P.bar_off = (P.r_off + red_bytes_rt(MT, CN) + 15) & ~15u;
  const uint32_t smem = P.bar_off + 16 * c.stages + 16 + 1024;  // + alignment slack
  if (smem > 227 * 1024) return TM_ERR_UNSUPPORTED;
  tm_status st;
  switch (MT) {
    case 1: st = launch_m<1>(c.tile_n, L.UPS, tmX, P, S, smem, stream); break;
    case 2: st = launch_m<2>(c.tile_n, L.UPS, tmX, P, S, smem, stream); break;
    case 4: st = launch_m<4>(c.tile_n, L.UPS, tmX, P, S, smem, stream); break;
    case 8: st = launch_m<8>(c.tile_n, L.UPS, tmX, P, S, smem, stream); break;
    default: return TM_ERR_UNSUPPORTED;
  }
  if (st == TM_OK) set_launch_count(1);
  return st;
}

}  // namespace w4
