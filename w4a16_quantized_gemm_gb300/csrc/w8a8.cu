// W8A8: 8-bit integer weights and activations ("LMDeploy Guide: Fast
// Mixed-Precision LLM Inference Engine": W8A8 among the served precision
// formats, produced by SmoothQuant-style post-training quantisation).
//
// Our reading, the SmoothQuant scheme in its plainest form (smoothing factors
// already folded into the fp16 weights):
//   activations per token (row m), dynamic and symmetric, weights per output
//   channel (column n), symmetric, each in IEEE binary32 with
//   round-to-nearest-even:
//     a = max |x|;  s = a / 127, or 1 when a == 0;  i = 1 / s;
//     q = clamp(rint(x * i), -127, 127)
//   Y[m][n] = s_x[m] s_w[n] sum_k q_x[m][k] q_w[k][n]
//
// GB300 design.  The int8 tensor-core rate of this part is far below its fp16
// rate, so both operands are turned into exact fp16 integers in registers
// (a byte OR-ed under the fp16 pattern of 1024 is 1024 + b; minus 1152 gives
// the signed value) and multiplied on mma.m16n8k16 with fp32 accumulation:
// every product is exact, and so is every partial sum below 2^24.  Weights
// stream through a shared-memory ring by bulk copies (one producer warp),
// X by 2-D TMA loads with the 128-byte swizzle; split-K CTAs of a thread-block
// cluster reduce through distributed shared memory; the epilogue applies
// s_x[m] s_w[n] and rounds to fp16 once.
//
// Packed weights (ours): W^T in blocks of 128 k, [Kp/128][N][128 bytes] --
// row n of a block holds the codes (biased: q + 128) of column n for those
// 128 k, K padded to Kp, a multiple of 128, with zero codes.  The kernels load
// 128 rows (8 n-tiles) of a block with one TMA box and the 128-byte swizzle
// (16-byte chunk c of row r stored at c ^ (r & 7)), which makes both reads
// conflict-free: the mma.sync path takes, for lane 4 gr + t, the 16 bytes at
// k 16t of rows gr and gr + 8 -- word st of each is the step-st A fragment
// once the step's k order is permuted the same way on X (slots 2t, 2t+1, 2t+8,
// 2t+9 -> k 16t + 4st + 0..3), so a lane's B fragments for a 64-k unit are the
// 16 bytes at 16t of an X row; the tensor-memory path has each thread convert
// its own row.
#include <algorithm>
#include <new>

#include "tm_common.cuh"
#include "../../include/tm_w8a8.h"

struct tm_w8_packed {
  int K, N, Kp, NT, KB;
  int device;
  uint8_t* codes;  // [KB][N][128]
  float* scales;   // [N]
  void* base;
  size_t bytes;
  CUtensorMap tm_codes;  // u8 {128, N, KB}, box {128, 128, 1}, 128-byte swizzle
};

namespace w4 {

namespace {

__device__ uint32_t s_err_w8;

constexpr int kW8Block = 2048;  // code bytes of one n-tile x 128 k
constexpr int kW8WN = 2;        // n-tiles per consumer warp
constexpr int kW8NW = 4;        // consumer warps
constexpr int kW8CN = kW8WN * kW8NW;
constexpr uint32_t kW8SmemMax = 227 * 1024;

// ---------------------------------------------------------- quantisers -----

// One CTA per row of X [M][K] (K % 8 == 0): the row's max |x|, then the codes.
// Under programmatic dependent launch the next grid (the GEMM, which streams
// its weights first) may start at once; X is read and xq, sx written only
// after the preceding grid finished.
__global__ void __launch_bounds__(256) w8_quant_act_kernel(const __half* __restrict__ X, int K,
                                                            int8_t* __restrict__ q, float* __restrict__ sx) {
  __shared__ float red[8];
  launch_dependents();
  grid_dependency_wait();
  const int m = blockIdx.x;
  const uint4* row = reinterpret_cast<const uint4*>(X + (size_t)m * K);
  const int nv = K / 8;
  float a = 0.f;
  for (int i = threadIdx.x; i < nv; i += 256) {
    const uint4 v = row[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
      a = fmaxf(a, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  a = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) a = fmaxf(a, red[w]);
  const float s = a == 0.f ? 1.f : __fdiv_rn(a, 127.f);
  const float inv = __fdiv_rn(1.f, s);
  if (threadIdx.x == 0) sx[m] = s;
  uint2* out = reinterpret_cast<uint2*>(q + (size_t)m * K);
  for (int i = threadIdx.x; i < nv; i += 256) {
    const uint4 v = row[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t b[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
      b[2 * e] = (uint32_t)(int)fminf(fmaxf(rintf(__fmul_rn(f.x, inv)), -127.f), 127.f) & 0xFFu;
      b[2 * e + 1] = (uint32_t)(int)fminf(fmaxf(rintf(__fmul_rn(f.y, inv)), -127.f), 127.f) & 0xFFu;
    }
    out[i] = make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24),
                        b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
  }
}

// ------------------------------------------------------------- packing -----

// One thread per 16-byte chunk of the packed codes: chunk c of row n of block
// kb holds the biased codes of column n at k = 128 kb + 16c .. +15.
__global__ void w8_pack_kernel(const int8_t* __restrict__ q, int K, int N, long long chunks, uint4* __restrict__ out) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= chunks) return;
  const int c = (int)(idx & 7);
  const long long row = idx >> 3;  // kb * N + n
  const int n = (int)(row % N), kb = (int)(row / N);
  uint32_t w[4];
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
    uint32_t v = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = kb * 128 + 16 * c + 4 * wi + j;
      const int code = k < K ? (int)q[(size_t)k * N + n] : 0;
      v |= (uint32_t)((code + 128) & 0xFF) << (8 * j);
    }
    w[wi] = v;
  }
  out[idx] = make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void w8_unpack_kernel(const uint8_t* __restrict__ codes, int K, int N, int8_t* __restrict__ q) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)K * N) return;
  const int k = (int)(idx / N), n = (int)(idx % N);
  q[idx] = (int8_t)((int)codes[((size_t)(k / 128) * N + n) * 128 + (k & 127)] - 128);
}

// --------------------------------------------------------------- GEMM ------

struct W8Params {
  const uint8_t* codes;
  const float* sw;
  const float* sx;
  __half* Y;
  int M, N, NT;
  int kb_total, kb_per_cta;
  int stages;
  uint32_t x_bytes;     // bytes of X per stage (8 MT rows x 128)
  uint32_t stage_bytes;
  uint32_t r_off, bar_off;
};

// Two biased codes (bytes 2i, 2i+1 of w) -> two exact fp16 values b - 128.
__device__ __forceinline__ uint32_t biased_to_half2(uint32_t w, int i) {
  return hsub2_u32(__byte_perm(w, 0x6464u, i == 0 ? 0x4140u : 0x4342u), 0x64806480u);
}

__device__ __forceinline__ bool w8_drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) {
      atomicOr(&s_err_w8, kErrTimeout);
      return false;
    }
  }
  return true;
}

// MT: 8-row tiles of X per CTA (8 MT rows from row blockIdx.x * 8 MT).
template <int MT>
__global__ void __launch_bounds__((kW8NW + 1) * 32) w8_kernel(const __grid_constant__ CUtensorMap tmX,
                                                              const __grid_constant__ CUtensorMap tmW,
                                                              const W8Params P) {
  constexpr int CNN = kW8CN * 16;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;  // the 128-byte swizzle repeats every 1024 bytes
  uint8_t* smem = smem_raw + (base - raw_base);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * 8 * MT;
  const int nt0 = blockIdx.z * kW8CN;
  const int S = gridDim.y;
  const int kb_begin = blockIdx.y * P.kb_per_cta;
  const int nkb = max(0, min(P.kb_total, kb_begin + P.kb_per_cta) - kb_begin);
  const int stages = P.stages;
  const uint32_t bar_full = base + P.bar_off;
  const uint32_t bar_empty = bar_full + 8 * stages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P.bar_off + 16 * stages);
  float* red = reinterpret_cast<float*>(smem + P.r_off);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kW8NW);
    }
    *abort_flag = 0;
    fence_mbar_init();
    launch_dependents();
  }
  __syncthreads();
  if (S > 1) cluster_arrive_relaxed();

  if (warp == kW8NW) {
    // ---------------- producer: one elected thread ----------------
    if (lane == 0) {
      prefetch_tmap(&tmX);
      prefetch_tmap(&tmW);
      const uint32_t tx = P.x_bytes + kW8CN * kW8Block;  // boxes count in full, zero-filled past N and K
      auto issue_w = [&](int i) {
        tma_load_3d(base + (i % stages) * P.stage_bytes + P.x_bytes, &tmW, 0, nt0 * 16, kb_begin + i,
                    bar_full + 8 * (i % stages));
      };
      auto issue_x = [&](int i) {
        tma_load_2d(base + (i % stages) * P.stage_bytes, &tmX, (kb_begin + i) * 128, m0, bar_full + 8 * (i % stages));
      };
      // weights first: they do not depend on the preceding kernel; X does
      const int first = min(nkb, stages);
      for (int i = 0; i < first; ++i) {
        mbar_expect_tx(bar_full + 8 * i, tx);
        issue_w(i);
      }
      grid_dependency_wait();
      for (int i = 0; i < first; ++i) issue_x(i);
      int issued = first;
      for (int i = first; i < nkb; ++i) {
        const int slot = i % stages;
        if (!mbar_wait(bar_empty + 8 * slot, (uint32_t)(i / stages - 1) & 1u, abort_flag, &s_err_w8)) break;
        mbar_expect_tx(bar_full + 8 * slot, tx);
        issue_w(i);
        issue_x(i);
        issued = i + 1;
      }
      // never leave with copies in flight into this CTA's shared memory
      for (int i = max(0, issued - stages); i < issued; ++i) w8_drain(bar_full + 8 * (i % stages), (uint32_t)(i / stages) & 1u);
    }
    __syncwarp();
    if (S > 1) cluster_wait();
  } else {
    // ---------------- consumers: kW8WN n-tiles each ----------------
    const int gr = lane >> 2, t = lane & 3;
    float acc[kW8WN][MT][4];
#pragma unroll
    for (int j = 0; j < kW8WN; ++j)
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][m][e] = 0.f;

    for (int i = 0; i < nkb; ++i) {
      const int slot = i % stages;
      if (!mbar_wait(bar_full + 8 * slot, (uint32_t)(i / stages) & 1u, abort_flag, &s_err_w8)) break;
      const uint8_t* stg = smem + (size_t)slot * P.stage_bytes;
      const uint8_t* cs = stg + P.x_bytes;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        // X row mt * 8 + gr, 16 bytes at k 64u + 16t (chunk 4u + t, swizzled by the row)
        uint32_t xw[MT][4];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const uint4 v = *reinterpret_cast<const uint4*>(stg + (m * 8 + gr) * 128 + (((4 * u + t) ^ gr) << 4));
          xw[m][0] = v.x ^ 0x80808080u;  // signed -> biased
          xw[m][1] = v.y ^ 0x80808080u;
          xw[m][2] = v.z ^ 0x80808080u;
          xw[m][3] = v.w ^ 0x80808080u;
        }
        // rows gr and gr + 8 of each n-tile, 16 bytes at k 64u + 16t (swizzled by the row)
        uint4 wg[kW8WN], wg8[kW8WN];
#pragma unroll
        for (int j = 0; j < kW8WN; ++j) {
          const uint8_t* r0 = cs + ((warp * kW8WN + j) * 16 + gr) * 128 + (((4 * u + t) ^ gr) << 4);
          wg[j] = *reinterpret_cast<const uint4*>(r0);
          wg8[j] = *reinterpret_cast<const uint4*>(r0 + 8 * 128);
        }
#pragma unroll
        for (int st = 0; st < 4; ++st) {
          uint32_t a[kW8WN][4];
#pragma unroll
          for (int j = 0; j < kW8WN; ++j) {
            const uint32_t w0 = st == 0 ? wg[j].x : st == 1 ? wg[j].y : st == 2 ? wg[j].z : wg[j].w;
            const uint32_t w8 = st == 0 ? wg8[j].x : st == 1 ? wg8[j].y : st == 2 ? wg8[j].z : wg8[j].w;
            a[j][0] = biased_to_half2(w0, 0);
            a[j][1] = biased_to_half2(w8, 0);
            a[j][2] = biased_to_half2(w0, 1);
            a[j][3] = biased_to_half2(w8, 1);
          }
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const uint32_t b0 = biased_to_half2(xw[m][st], 0), b1 = biased_to_half2(xw[m][st], 1);
#pragma unroll
            for (int j = 0; j < kW8WN; ++j) mma_16816(acc[j][m], a[j], b0, b1);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
    }

    // Partial tile -> the owner of each column slice: red[rank][m][col] in
    // the owner's shared memory (its own when S == 1).
    const int span = CNN / S;
    const uint32_t my_rank = S > 1 ? cluster_ctarank() : 0u;
    const uint32_t red_s = smem_u32(red);
    if (S > 1) cluster_wait();
#pragma unroll
    for (int j = 0; j < kW8WN; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int nl = (warp * kW8WN + j) * 16 + gr + ((e & 2) ? 8 : 0);
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

  // ---------------- reduction of this CTA's column slice, scaling ----------------
  if (S > 1) {
    cluster_sync_all();
  } else {
    __syncthreads();
  }
  grid_dependency_wait();  // Y may still be read by the preceding grid
  const int span = CNN / S;
  const uint32_t my_rank = S > 1 ? cluster_ctarank() : 0u;
  const int half_span = span >> 1;
  const int n_base = nt0 * 16 + (int)my_rank * span;
  const int rows = min(8 * MT, P.M - m0);
  for (int it = threadIdx.x; it < rows * half_span; it += blockDim.x) {
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
    const float s = P.sx[m0 + m];
    const float2 w = *reinterpret_cast<const float2*>(P.sw + n);
    *reinterpret_cast<__half2*>(P.Y + (size_t)(m0 + m) * P.N + n) = __floats2half2_rn(v.x * s * w.x, v.y * s * w.y);
  }
}

int w8_mt(int M) { return M <= 8 ? 1 : M <= 16 ? 2 : M <= 32 ? 4 : 8; }

struct W8Shape {
  uint32_t x_bytes, stage, red;
};

W8Shape w8_shape(int MT) {
  W8Shape g;
  g.x_bytes = (uint32_t)MT * 1024u;
  g.stage = (g.x_bytes + kW8CN * kW8Block + 1023u) & ~1023u;
  g.red = (uint32_t)MT * 8 * kW8CN * 16 * 4;
  return g;
}

uint32_t w8_smem(const W8Shape& g, int stages) {
  const uint32_t bar_off = (g.stage * stages + g.red + 15u) & ~15u;
  return bar_off + 16 * stages + 16 + 1024;  // + alignment slack
}

template <int MT>
tm_status w8_launch_t(const CUtensorMap& tmX, const CUtensorMap& tmW, const W8Params& P, dim3 grid, int S,
                      uint32_t smem, cudaStream_t stream) {
  auto kern = w8_kernel<MT>;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kW8SmemMax) != cudaSuccess)
      return TM_ERR_CUDA;
    attr_done = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3((kW8NW + 1) * 32, 1, 1);
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
  return cudaLaunchKernelEx(&cfg, kern, tmX, tmW, P) == cudaSuccess ? TM_OK : TM_ERR_CUDA;
}

unsigned grid_1d(long long n, int block) { return (unsigned)((n + block - 1) / block); }

}  // namespace

cudaError_t w8_error_bits(uint32_t* bits, bool clear) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, s_err_w8, sizeof(v));
  if (e != cudaSuccess) return e;
  if (clear && v) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(s_err_w8, &zero, sizeof(zero));
  }
  *bits = v;
  return e;
}

}  // namespace w4

using namespace w4;

extern "C" tm_status tm_w8a8_quantize_act(const uint16_t* X, int M, int K, int8_t* xq, float* sx, void* stream) {
  if (!X || !xq || !sx || M < 0 || K <= 0 || K % 16) return TM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(X) & 15u) || (reinterpret_cast<uintptr_t>(xq) & 15u) ||
      (reinterpret_cast<uintptr_t>(sx) & 3u))
    return TM_ERR_ALIGNMENT;
  if (M == 0) return TM_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)M, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, w8_quant_act_kernel, reinterpret_cast<const __half*>(X), K, xq, sx) != cudaSuccess)
    return TM_ERR_CUDA;
  set_launch_count(1);
  return TM_OK;
}

extern "C" tm_status tm_w8_pack(const int8_t* q, const float* sw, int K, int N, tm_w8_packed** out) {
  if (!out) return TM_ERR_INVALID_ARG;
  *out = nullptr;
  if (!q || !sw || K <= 0 || N <= 0 || K % 16 || N % 16) return TM_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TM_ERR_CUDA;
  tm_w8_packed* p = new (std::nothrow) tm_w8_packed;
  if (!p) return TM_ERR_CUDA;
  p->K = K;
  p->N = N;
  p->Kp = (K + 127) / 128 * 128;
  p->NT = N / 16;
  p->KB = p->Kp / 128;
  p->device = dev;
  const size_t code_bytes = (size_t)p->KB * N * 128;
  p->bytes = code_bytes + (size_t)N * 4;
  if (cudaMalloc(&p->base, p->bytes) != cudaSuccess) {
    delete p;
    return TM_ERR_CUDA;
  }
  p->codes = static_cast<uint8_t*>(p->base);
  p->scales = reinterpret_cast<float*>(p->codes + code_bytes);
  {
    EncodeTiledFn fn = encode_tiled_fn();
    cuuint64_t dims[3] = {128, (cuuint64_t)N, (cuuint64_t)p->KB};
    cuuint64_t strides[2] = {128, (cuuint64_t)N * 128};
    cuuint32_t box[3] = {128, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (!fn || fn(&p->tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, p->codes, dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      cudaFree(p->base);
      delete p;
      return TM_ERR_CUDA;
    }
  }
  const long long chunks = (long long)code_bytes / 16;
  w8_pack_kernel<<<grid_1d(chunks, 256), 256>>>(q, K, N, chunks, reinterpret_cast<uint4*>(p->codes));
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaMemcpy(p->scales, sw, (size_t)N * 4, cudaMemcpyDeviceToDevice);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(p->base);
    delete p;
    return TM_ERR_CUDA;
  }
  *out = p;
  return TM_OK;
}

extern "C" tm_status tm_w8_unpack(const tm_w8_packed* p, int8_t* q, float* sw) {
  if (!p || !q || !sw) return TM_ERR_INVALID_ARG;
  w8_unpack_kernel<<<grid_1d((long long)p->K * p->N, 256), 256>>>(p->codes, p->K, p->N, q);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaMemcpy(sw, p->scales, (size_t)p->N * 4, cudaMemcpyDeviceToDevice);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return e == cudaSuccess ? TM_OK : TM_ERR_CUDA;
}

extern "C" tm_status tm_w8_packed_info(const tm_w8_packed* p, int* K, int* N, size_t* bytes) {
  if (!p) return TM_ERR_INVALID_ARG;
  if (K) *K = p->K;
  if (N) *N = p->N;
  if (bytes) *bytes = p->bytes;
  return TM_OK;
}

extern "C" void tm_w8_packed_free(tm_w8_packed* p) {
  if (!p) return;
  cudaFree(p->base);
  delete p;
}

extern "C" tm_status tm_w8a8_gemm(const int8_t* xq, const float* sx, const tm_w8_packed* p, void* Y, int M,
                                  int split_k, void* stream) {
  if (!xq || !sx || !p || !Y || M < 0) return TM_ERR_INVALID_ARG;
  if (split_k < 0 || split_k > 8 || (split_k & (split_k - 1))) return TM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(xq) & 15u) || (reinterpret_cast<uintptr_t>(Y) & 15u) ||
      (reinterpret_cast<uintptr_t>(sx) & 3u))
    return TM_ERR_ALIGNMENT;
  if (M == 0) return TM_OK;
  const int MT = w8_mt(M);
  const int MB = (M + 8 * MT - 1) / (8 * MT);
  const int NB = (p->NT + kW8CN - 1) / kW8CN;
  // the smallest split (a cluster along K) giving 256 CTAs, each with at least
  // two 128-k blocks
  int S = split_k;
  if (!S) {
    S = 1;
    while (S < 8 && (long long)NB * MB * S < 256 && p->KB / (2 * S) >= 2) S *= 2;
  }
  const W8Shape g = w8_shape(MT);
  int per_sm = 0, reserved = 0;
  sm_shared_memory(p->device, &per_sm, &reserved);
  const long long ctas = (long long)NB * MB * S;
  const int sms = num_sms(p->device);
  const int r = (int)std::max<long long>(1, (ctas + sms - 1) / sms);
  const uint32_t budget = (uint32_t)std::min<int>((int)kW8SmemMax, std::max(0, per_sm / r - reserved)) & ~127u;
  const int kb_per_cta = (p->KB + S - 1) / S;
  int stages = 8;
  while (stages > 2 && w8_smem(g, stages) > budget) --stages;
  stages = std::max(2, std::min(stages, std::max(2, kb_per_cta)));
  const uint32_t need = w8_smem(g, stages);
  if (need > kW8SmemMax) return TM_ERR_UNSUPPORTED;
  const uint32_t smem = std::max(need, budget);

  CUtensorMap tmX;
  {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return TM_ERR_CUDA;
    cuuint64_t dims[2] = {(cuuint64_t)p->K, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)p->K};
    cuuint32_t box[2] = {128, (cuuint32_t)(8 * MT)};
    cuuint32_t es[2] = {1, 1};
    if (fn(&tmX, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(xq), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return TM_ERR_CUDA;
  }
  W8Params P;
  P.codes = p->codes;
  P.sw = p->scales;
  P.sx = sx;
  P.Y = reinterpret_cast<__half*>(Y);
  P.M = M;
  P.N = p->N;
  P.NT = p->NT;
  P.kb_total = p->KB;
  P.kb_per_cta = kb_per_cta;
  P.stages = stages;
  P.x_bytes = g.x_bytes;
  P.stage_bytes = g.stage;
  P.r_off = g.stage * stages;
  P.bar_off = (P.r_off + g.red + 15u) & ~15u;
  const dim3 grid((unsigned)MB, (unsigned)S, (unsigned)NB);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  tm_status res = TM_ERR_UNSUPPORTED;
  switch (MT) {
    case 1: res = w8_launch_t<1>(tmX, p->tm_codes, P, grid, S, smem, st); break;
    case 2: res = w8_launch_t<2>(tmX, p->tm_codes, P, grid, S, smem, st); break;
    case 4: res = w8_launch_t<4>(tmX, p->tm_codes, P, grid, S, smem, st); break;
    case 8: res = w8_launch_t<8>(tmX, p->tm_codes, P, grid, S, smem, st); break;
    default: break;
  }
  if (res == TM_OK) set_launch_count(1);
  return res;
}
