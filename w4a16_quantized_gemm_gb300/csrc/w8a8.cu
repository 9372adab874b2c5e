// W8A8: 8-bit integer weights and activations ("LMDeploy Guide: Fast
// Mixed-Precision LLM Inference Engine": W8A8 among the served precision
// formats, produced by SmoothQuant-style post-training quantisation).
//
// Our reading, the SmoothQuant scheme in its plainest form (smoothing factors
// already folded into the fp16 weights):
//   activations per token (row m), dynamic and symmetric, weights per output
//   channel (column n), symmetric, each in IEEE binary32 with
//   round-to-nearest-even:
//     a = max |x|;  s = a / 127, or 1 when a == 0;
//     q = clamp(rint(x / s), -127, 127)     (an IEEE division per value: s is
//     a binary32 value, and x * (1/s) can round a code differently)
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
// F16: the codes written as exact fp16 integers (for the tensor-memory
// kernel's X path), else as int8.
template <bool F16>
__global__ void __launch_bounds__(256) w8_quant_act_kernel(const __half* __restrict__ X, int K,
                                                            void* __restrict__ q, float* __restrict__ sx) {
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
  if (threadIdx.x == 0) sx[m] = s;
  for (int i = threadIdx.x; i < nv; i += 256) {
    const uint4 v = row[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float c[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
      c[2 * e] = fminf(fmaxf(rintf(__fdiv_rn(f.x, s)), -127.f), 127.f);
      c[2 * e + 1] = fminf(fmaxf(rintf(__fdiv_rn(f.y, s)), -127.f), 127.f);
    }
    if (F16) {
      // integers of magnitude <= 127: exact in fp16
      uint32_t h[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __half2 t = __floats2half2_rn(c[2 * e], c[2 * e + 1]);
        h[e] = *reinterpret_cast<const uint32_t*>(&t);
      }
      reinterpret_cast<uint4*>(static_cast<__half*>(q) + (size_t)m * K)[i] = make_uint4(h[0], h[1], h[2], h[3]);
    } else {
      uint32_t b[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) b[e] = (uint32_t)(int)c[e] & 0xFFu;
      reinterpret_cast<uint2*>(static_cast<int8_t*>(q) + (size_t)m * K)[i] =
          make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24), b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
    }
  }
}

// Per-channel weight quantisation, three launches after zeroing sw: the column
// maxima of |w| (a block per 256 columns x a slice of K, combined with an
// integer atomic max -- the patterns of non-negative floats order like the
// floats), then the codes with s = max / 127 recomputed per block, then sw
// itself in place.
constexpr int kWqRows = 512;  // rows of K per block

__global__ void __launch_bounds__(256) w8_colmax_kernel(const __half* __restrict__ W, int K, int N,
                                                         uint32_t* __restrict__ amax) {
  __shared__ float red[8][32][8];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int c8 = blockIdx.x * 32 + tx, N8 = N / 8;
  const int k0 = blockIdx.y * kWqRows, k1 = min(K, k0 + kWqRows);
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (c8 < N8) {
    for (int k = k0 + ty; k < k1; k += 8) {
      const uint4 v = *reinterpret_cast<const uint4*>(W + (size_t)k * N + 8 * c8);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
        a[2 * e] = fmaxf(a[2 * e], fabsf(f.x));
        a[2 * e + 1] = fmaxf(a[2 * e + 1], fabsf(f.y));
      }
    }
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) red[ty][tx][c] = a[c];
  __syncthreads();
  if (ty == 0 && c8 < N8) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float m = red[0][tx][c];
#pragma unroll
      for (int y = 1; y < 8; ++y) m = fmaxf(m, red[y][tx][c]);
      atomicMax(amax + 8 * c8 + c, __float_as_uint(m));
    }
  }
}

__device__ __forceinline__ float w8_scale_of(uint32_t amax_bits) {
  const float a = __uint_as_float(amax_bits);
  return a == 0.f ? 1.f : __fdiv_rn(a, 127.f);
}

__global__ void __launch_bounds__(256) w8_wquant_kernel(const __half* __restrict__ W, int K, int N,
                                                         const uint32_t* __restrict__ amax, int8_t* __restrict__ q) {
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int c8 = blockIdx.x * 32 + tx, N8 = N / 8;
  if (c8 >= N8) return;
  const int k0 = blockIdx.y * kWqRows, k1 = min(K, k0 + kWqRows);
  float sc[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) sc[c] = w8_scale_of(amax[8 * c8 + c]);
  for (int k = k0 + ty; k < k1; k += 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(W + (size_t)k * N + 8 * c8);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t b[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
      b[2 * e] = (uint32_t)(int)fminf(fmaxf(rintf(__fdiv_rn(f.x, sc[2 * e])), -127.f), 127.f) & 0xFFu;
      b[2 * e + 1] = (uint32_t)(int)fminf(fmaxf(rintf(__fdiv_rn(f.y, sc[2 * e + 1])), -127.f), 127.f) & 0xFFu;
    }
    *reinterpret_cast<uint2*>(q + (size_t)k * N + 8 * c8) =
        make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24), b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
  }
}

__global__ void w8_scale_kernel(float* __restrict__ sw, int N) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n < N) sw[n] = w8_scale_of(__float_as_uint(sw[n]));
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

// ---------------------------------------------- tensor-memory W8A8 GEMM -----
//
// For larger M the products go to tcgen05 (kind::f16, fp32 accumulators in
// tensor memory), both operands as exact fp16 integers:
//   * warp 0, one thread: per 128-k block one TMA box of weight codes (128
//     rows of W^T = the CTA's 128 output columns) and one of X (BT rows), both
//     with the 128-byte swizzle, into a ring; weights of the first slots before
//     `griddepcontrol.wait`, X after;
//   * warps 2..9 convert a ring slot into one of the "converted" slots: the
//     warp pair of tensor-memory lane quarter q turns rows 32q .. 32q+31 of the
//     weight box (one 64-k unit each) into fp16 and writes them with
//     tcgen05.st.32x32b as the MMA's A operand (lane = output column, column c
//     = k pair c of a 16-k slice); with int8 X all 256 threads also turn the X
//     box into fp16 rows of 128 bytes with the 128-byte swizzle (the K-major B
//     operand); then they release the ring slot;
//   * with X given as fp16 codes, X has a ring of its own, one 64-k unit (BT
//     rows x 128 bytes) per slot, each freed by the commit of the MMAs that
//     read it, so that a weight slot is free as soon as it is converted (three
//     weight slots, five X units and four tensor-memory A slots at 256-row
//     tiles; one ring of two 80 KB slots held X and weights before);
//   * warp 1, one thread: 8 MMAs (M = 128, N = BT, K = 16) per converted slot,
//     whose commit frees it;
//   * warps 2..9 again: epilogue, y = acc s_x[m] s_w[n] -> fp16; split K over a
//     cluster reduces through distributed shared memory in rank order.
constexpr int kW8TcThreads = 320;
constexpr int kW8TcConv = 2;  // converted slots with int8 X (tensor-memory A + fp16 X in shared memory)

template <int BT, bool XH>
struct W8TcShape {
  static constexpr uint32_t W_BYTES = 128 * 128;  // one 128-k block of 128 weight rows
  static constexpr uint32_t XR_BYTES = BT * 128;  // one 128-k block of BT int8 rows
  static constexpr uint32_t XF_UNIT = BT * 128;   // fp16 X, one 64-k unit
  static constexpr uint32_t XF_SLOT = 2 * XF_UNIT;
  // XH: X arrives as fp16 codes in a ring of its own, one 64-k unit per slot,
  // each freed by the MMAs' commit, while the weight ring's slots are freed
  // as soon as they are converted; otherwise X arrives as int8 next to the
  // weights and is converted into XF_SLOT-sized buffers of its own.
  static constexpr uint32_t SLOT = W_BYTES + (XH ? 0 : XR_BYTES);
  static constexpr uint32_t CONV_SLOTS = XH ? 0 : kW8TcConv;  // converted X buffers
  // converted slots: with fp16 X only tensor-memory A slots, four of them
  static constexpr int SC = XH ? 4 : kW8TcConv;
  static constexpr uint32_t A_COLS = 64;  // 8 slices of 16 k, 8 columns each
  static constexpr uint32_t A_COL = BT;   // A slots right after the accumulator columns
  static constexpr uint32_t TMEM_COLS = BT + SC * A_COLS <= 256 ? 256 : 512;
  static_assert(BT + SC * A_COLS <= 512, "tensor memory");
  static constexpr int TPR = 256 / BT;     // converter threads per X row
  static constexpr int CPT = 8 / TPR;      // 16-byte X chunks per converter thread
  static_assert(SLOT % 1024 == 0 && XF_UNIT % 1024 == 0, "swizzled tiles need 1024-byte alignment");
};

struct W8TcParams {
  const float* sw;
  const float* sx;
  __half* Y;
  int M, N;
  int kb_total, kb_per_cta;
  int stages;       // ring slots
  int xstages;      // XH: slots of the X ring (64-k units)
  uint32_t x_off;   // XH: offset of the X ring
  uint32_t xf_off;  // offset of the converted X slots
  uint32_t bar_off;
};

__device__ __forceinline__ void tc_st_32x32b_x8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]));
}

template <int BT, bool XH>
__global__ void __launch_bounds__(kW8TcThreads, 1)
    w8tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                const __grid_constant__ CUtensorMap tmY, const W8TcParams P) {
  using SH = W8TcShape<BT, XH>;
  constexpr int SC = SH::SC;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_base);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // row blocks vary fastest: the CTAs that share a weight tile run together
  // and read it from L2
  const int m0 = blockIdx.x * BT;
  const int nt0 = blockIdx.y * 8;
  const int S = gridDim.z;
  const int kb0 = blockIdx.z * P.kb_per_cta;
  const int nkb = max(0, min(P.kb_total, kb0 + P.kb_per_cta) - kb0);
  const int SA = P.stages;
  const int SX = XH ? P.xstages : 0;

  const uint32_t barA = base + P.bar_off;  // [SA] full, then [SA] empty
  const uint32_t barC = barA + 16 * SA;    // [SC] full, then [SC] empty (converted slots)
  const uint32_t barX = barC + 16 * SC;    // XH: [SX] full, then [SX] empty (X units)
  const uint32_t bar_acc = barX + 16 * SX;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + P.bar_off + 16 * (SA + SC + SX) + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P.bar_off + 16 * (SA + SC + SX) + 12);
  auto fullA = [&](int s) { return barA + 8 * s; };
  auto emptyA = [&](int s) { return barA + 8 * (SA + s); };
  auto fullC = [&](int s) { return barC + 8 * s; };
  auto emptyC = [&](int s) { return barC + 8 * (SC + s); };
  auto fullX = [&](int s) { return barX + 8 * s; };
  auto emptyX = [&](int s) { return barX + 8 * (SX + s); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < SA; ++s) {
      mbar_init(fullA(s), 1);
      mbar_init(emptyA(s), 8);  // freed by the eight converter warps
    }
    for (int s = 0; s < SC; ++s) {
      mbar_init(fullC(s), 8);
      mbar_init(emptyC(s), 1);
    }
    for (int s = 0; s < SX; ++s) {
      mbar_init(fullX(s), 1);
      mbar_init(emptyX(s), 1);  // freed by the commit of the MMAs that read it
    }
    mbar_init(bar_acc, 1);
    *abort_flag = 0;
    fence_mbar_init();
    launch_dependents();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), SH::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // D at columns 0 .. BT-1, A slots from A_COL

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tmap(&tmX);
      prefetch_tmap(&tmW);
      auto issue_w = [&](int i, int s) { tma_load_3d(base + s * SH::SLOT, &tmW, 0, nt0 * 16, kb0 + i, fullA(s)); };
      const int first = min(nkb, SA);
      for (int i = 0; i < first; ++i) {
        mbar_expect_tx(fullA(i), SH::SLOT);
        issue_w(i, i);
      }
      grid_dependency_wait();
      int issued = first, issued_x = 0;
      if constexpr (XH) {
        // in the order the MMAs consume them: block i's weights, then its two X units
        auto issue_xu = [&](int j) {
          const int sx = j % SX;
          if (j >= SX && !mbar_wait(emptyX(sx), (uint32_t)(j / SX - 1) & 1u, abort_flag, &s_err_w8)) return false;
          mbar_expect_tx(fullX(sx), SH::XF_UNIT);
          tma_load_2d(base + P.x_off + sx * SH::XF_UNIT, &tmX, kb0 * 128 + 64 * j, m0, fullX(sx));
          issued_x = j + 1;
          return true;
        };
        bool ok = true;
        for (int i = 0; i < nkb && ok; ++i) {
          if (i >= first) {
            const int s = i % SA;
            if (!mbar_wait(emptyA(s), (uint32_t)(i / SA - 1) & 1u, abort_flag, &s_err_w8)) break;
            mbar_expect_tx(fullA(s), SH::SLOT);
            issue_w(i, s);
            issued = i + 1;
          }
          ok = issue_xu(2 * i) && issue_xu(2 * i + 1);
        }
        for (int j = max(0, issued_x - SX); j < issued_x; ++j) w8_drain(fullX(j % SX), (uint32_t)(j / SX) & 1u);
      } else {
        for (int i = 0; i < first; ++i) tma_load_2d(base + i * SH::SLOT + SH::W_BYTES, &tmX, (kb0 + i) * 128, m0, fullA(i));
        for (int i = first; i < nkb; ++i) {
          const int s = i % SA;
          if (!mbar_wait(emptyA(s), (uint32_t)(i / SA - 1) & 1u, abort_flag, &s_err_w8)) break;
          mbar_expect_tx(fullA(s), SH::SLOT);
          issue_w(i, s);
          tma_load_2d(base + s * SH::SLOT + SH::W_BYTES, &tmX, (kb0 + i) * 128, m0, fullA(s));
          issued = i + 1;
        }
      }
      // never leave with copies in flight into this CTA's shared memory
      for (int i = max(0, issued - SA); i < issued; ++i) w8_drain(fullA(i % SA), (uint32_t)(i / SA) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(128, BT);
      for (int i = 0; i < nkb; ++i) {
        const int sc = i % SC;
        if (!mbar_wait(fullC(sc), (uint32_t)(i / SC) & 1u, abort_flag, &s_err_w8)) break;
        const uint32_t ta = tmem + SH::A_COL + SH::A_COLS * sc;
        bool ok = true;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          uint64_t db;
          if constexpr (XH) {
            // B: the fp16 X of unit 2i + u in the X ring
            const int j = 2 * i + u, sx = j % SX;
            if (!mbar_wait(fullX(sx), (uint32_t)(j / SX) & 1u, abort_flag, &s_err_w8)) {
              ok = false;
              break;
            }
            tc_fence_after();
            db = smem_desc_sw128(base + P.x_off + sx * SH::XF_UNIT);
          } else {
            tc_fence_after();
            db = smem_desc_sw128(base + P.xf_off + sc * SH::XF_SLOT) + (uint64_t)((u * SH::XF_UNIT) >> 4);
          }
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc_mma_f16_ta(tmem, ta + 8u * (4 * u + k), db + (uint64_t)(2 * k), idesc, (i > 0 || u > 0 || k > 0) ? 1u : 0u);
          if constexpr (XH) tc_commit(emptyX((2 * i + u) % SX));
        }
        if (!ok) break;
        tc_commit(emptyC(sc));
      }
      // completes once every MMA issued above has finished (also on abort)
      tc_commit(bar_acc);
    }
    __syncwarp();
  } else {
    // ---------------- converters: warps 2..9 ----------------
    const int cw = warp - 2;
    const int q = warp & 3;    // tensor-memory lane quarter of this warp
    const int hu = cw >> 2;    // its 64-k unit of the weight block
    const int wrow = 32 * q + lane;
    const uint32_t t_lane = (uint32_t)(32 * q) << 16;
    const int T = cw * 32 + lane;
    const int xr = T / SH::TPR, part = T % SH::TPR;
    for (int i = 0; i < nkb; ++i) {
      const int s = i % SA, sc = i % SC;
      if (!mbar_wait(fullA(s), (uint32_t)(i / SA) & 1u, abort_flag, &s_err_w8)) break;
      if (!mbar_wait(emptyC(sc), ((uint32_t)(i / SC) & 1u) ^ 1u, abort_flag, &s_err_w8)) break;
      tc_fence_after();
      const uint32_t st = base + s * SH::SLOT;
      // weights: row wrow, k 64 hu + 16 s4 .. +15 -> 8 columns of slice 4 hu + s4
#pragma unroll
      for (int s4 = 0; s4 < 4; ++s4) {
        const uint4 v = lds128(st + wrow * 128 + (((4 * hu + s4) ^ (wrow & 7)) << 4));
        const uint32_t r[8] = {biased_to_half2(v.x, 0), biased_to_half2(v.x, 1), biased_to_half2(v.y, 0),
                               biased_to_half2(v.y, 1), biased_to_half2(v.z, 0), biased_to_half2(v.z, 1),
                               biased_to_half2(v.w, 0), biased_to_half2(v.w, 1)};
        tc_st_32x32b_x8(tmem + t_lane + SH::A_COL + SH::A_COLS * sc + 8u * (4 * hu + s4), r);
      }
      // X: row xr, chunks part * CPT .. +CPT-1 (16 k each) -> fp16, 128-byte swizzle
      const uint32_t xin = st + SH::W_BYTES + xr * 128;
      const uint32_t xout = base + P.xf_off + sc * SH::XF_SLOT + xr * 128;
#pragma unroll
      for (int c2 = 0; c2 < (XH ? 0 : SH::CPT); ++c2) {
        const int c = part * SH::CPT + c2;
        const uint4 v = lds128(xin + ((c ^ (xr & 7)) << 4));
        const uint32_t w0 = v.x ^ 0x80808080u, w1 = v.y ^ 0x80808080u, w2 = v.z ^ 0x80808080u,
                       w3 = v.w ^ 0x80808080u;
        const uint32_t o = xout + (c >> 2) * SH::XF_UNIT;
        const int oc = 2 * (c & 3);
        sts128(o + ((oc ^ (xr & 7)) << 4), biased_to_half2(w0, 0), biased_to_half2(w0, 1), biased_to_half2(w1, 0),
               biased_to_half2(w1, 1));
        sts128(o + (((oc + 1) ^ (xr & 7)) << 4), biased_to_half2(w2, 0), biased_to_half2(w2, 1),
               biased_to_half2(w3, 0), biased_to_half2(w3, 1));
      }
      tc_wait_st();
      tc_fence_before();
      if (!XH) fence_proxy_async_smem();  // the fp16 X tile is read by the tensor core (async proxy)
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(fullC(sc));
        mbar_arrive(emptyA(s));
      }
    }
  }

  // ---------------- epilogue: warps 2..9, TMEM lanes 32 q .. 32 q + 31 ----------------
  const bool epi = warp >= 2;
  const int q = warp & 3;
  const int h = (warp - 2) >> 2;
  const int row = 32 * q + lane;  // output column within the CTA (TMEM lane)
  constexpr int HALF = BT / 2;    // token columns per epilogue warp
  bool acc_ok = true;
  // s_x of one tile row and s_w of this thread's column, loaded before the
  // accumulator is complete so that their latency hides under the last MMAs
  const int xrow = threadIdx.x - 64;
  const float sx_mine = epi && xrow < BT && m0 + xrow < P.M ? P.sx[m0 + xrow] : 0.f;
  const int n_mine = nt0 * 16 + row;
  const float sw_mine = epi && n_mine < P.N ? P.sw[n_mine] : 0.f;
  if (epi) {
    acc_ok = mbar_wait(bar_acc, 0, abort_flag, &s_err_w8);
    acc_ok = __all_sync(0xffffffffu, acc_ok);
    tc_fence_after();
  }
  if (S == 1) {
    // The ring is idle once the accumulator is complete (every copy was
    // consumed by an MMA): the scaled fp16 tile is staged there, rows of 128
    // columns (256 bytes), with s_x of the tile's rows after it, and leaves
    // in one TMA tensor store that clips rows past M and columns past N.
    const uint32_t ystage = base;
    float* sxs = reinterpret_cast<float*>(smem + BT * 256);
    if (epi) {
      if (xrow < BT) sxs[xrow] = sx_mine;  // BT <= 256 epilogue threads
      epilogue_sync();
    }
    if (epi && acc_ok) {
      const float swn = sw_mine;
      // 32 accumulator columns per wait (tcgen05.wait::ld waits for every load in flight)
#pragma unroll 1
      for (int c = 0; c < HALF; c += 32) {
        uint32_t v[32];
#pragma unroll
        for (int b = 0; b < 4; ++b)
          tc_ld_32x32b_x8(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(h * HALF + c + 8 * b),
                          *reinterpret_cast<uint32_t(*)[8]>(v + 8 * b));
        tc_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int ml = h * HALF + c + e;  // row within the tile
          sts16(ystage + ml * 256 + row * 2,
                __half_as_ushort(__float2half_rn(__uint_as_float(v[e]) * sxs[ml] * swn)));
        }
      }
    }
    if (epi) {
      fence_proxy_async_smem();  // the staged tile is read by the TMA (async proxy)
      epilogue_sync();
    }
    if (warp == 2 && lane == 0 && acc_ok) {
      grid_dependency_wait();  // Y may still be read by the preceding grid
      tma_store_2d(&tmY, ystage, nt0 * 16, m0);
      bulk_commit_group();
      bulk_wait_group_read0();  // the shared memory stays ours until the store has read it
    }
  } else {
    // Split K: every CTA's ring is idle once all of the cluster passes this
    // barrier (MMAs finished, copies drained), so partial tiles may land there.
    cluster_sync_all();
    const int R = 128 / S;  // output columns owned by each rank
    const uint32_t my_rank = cluster_ctarank();
    if (epi) {
      const int owner = row / R, rr = row - owner * R;
      const uint32_t dst = map_shared_rank(base + (uint32_t)(((int)my_rank * R + rr) * BT) * 4u, (uint32_t)owner);
#pragma unroll 1
      for (int c = 0; c < HALF; c += 8) {
        uint32_t v[8];
        if (acc_ok && nkb > 0) {  // a CTA with no K blocks contributes zeros
          tc_ld_32x32b_x8(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(h * HALF + c), v);
          tc_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = 0u;
        }
        const uint32_t d = dst + (uint32_t)(h * HALF + c) * 4u;
        st_dsmem_v4(d, v[0], v[1], v[2], v[3]);
        st_dsmem_v4(d + 16, v[4], v[5], v[6], v[7]);
      }
    }
    cluster_sync_all();
    grid_dependency_wait();
    const float* red = reinterpret_cast<const float*>(smem);
    const int n_base = nt0 * 16 + (int)my_rank * R;
    for (int it = threadIdx.x; it < R * BT; it += blockDim.x) {
      const int tok = it / R, rr = it - tok * R;
      const int m = m0 + tok, n = n_base + rr;
      if (m >= P.M || n >= P.N) continue;
      float acc = 0.f;
#pragma unroll 8
      for (int k = 0; k < S; ++k) acc += red[(k * R + rr) * BT + tok];
      P.Y[(size_t)m * P.N + n] = __float2half_rn(acc * P.sx[m] * P.sw[n]);
    }
  }
  if (warp == 1 && lane == 0) w8_drain(bar_acc, 0);  // no MMA may still run when TMEM is released
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, SH::TMEM_COLS);
  }
}

template <int BT, bool XH>
tm_status w8tc_launch_t(const CUtensorMap& tmX, const CUtensorMap& tmW, const CUtensorMap& tmY, const W8TcParams& P,
                        dim3 grid, int S, uint32_t smem, cudaStream_t stream) {
  auto kern = w8tc_kernel<BT, XH>;
  static std::atomic<unsigned long long> attr_done{0};  // one bit per device
  if (!smem_attr_once(attr_done, (const void*)kern, (int)kW8SmemMax)) return TM_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kW8TcThreads, 1, 1);
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
    at[na].val.clusterDim.y = 1;
    at[na].val.clusterDim.z = (unsigned)S;
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, tmX, tmW, tmY, P) == cudaSuccess ? TM_OK : TM_ERR_CUDA;
}

// Shared memory of the tensor-memory kernel: ring, converted X slots, barriers, alignment slack.
template <int BT, bool XH>
uint32_t w8tc_smem(int stages, int xstages) {
  using SH = W8TcShape<BT, XH>;
  return stages * SH::SLOT + xstages * SH::XF_UNIT + SH::CONV_SLOTS * SH::XF_SLOT +
         16 * (stages + SH::SC + xstages) + 16 + 1024;
}

// xq: int8 codes, or (XH) the same codes as fp16 integers.
template <int BT, bool XH>
tm_status w8tc_run(const void* xq, const float* sx, const tm_w8_packed* p, void* Y, int M, int split_k,
                   cudaStream_t stream) {
  using SH = W8TcShape<BT, XH>;
  const int NB = (p->NT + 7) / 8, MB = (M + BT - 1) / BT;
  const int sms = num_sms(p->device);
  int S = split_k;
  if (!S) {
    // split K (a cluster) while the doubled grid still fits in one wave (one
    // CTA per SM) and each CTA keeps at least two 128-k blocks
    S = 1;
    while (S < 8 && (long long)NB * MB * S * 2 <= sms && p->KB / (2 * S) >= 2) S *= 2;
  }
  // XH: three weight slots and as many 64-k X units as fit (at most 8; two
  // weight slots for a sixth X unit at 256-row tiles measured no faster);
  // otherwise as many combined slots as fit
  int stages = XH ? 3 : 8, xstages = XH ? 8 : 0;
  if (XH) {
    while (xstages > 2 && w8tc_smem<BT, XH>(stages, xstages) > kW8SmemMax) --xstages;
  } else {
    while (stages > 2 && w8tc_smem<BT, XH>(stages, 0) > kW8SmemMax) --stages;
  }
  const uint32_t smem = w8tc_smem<BT, XH>(stages, xstages);
  if (smem > kW8SmemMax) return TM_ERR_UNSUPPORTED;
  // split K reduces through the shared memory below the barriers: S x (128 / S) columns x BT rows of fp32
  if (S > 1 && (uint32_t)128 * BT * 4 >
                   stages * SH::SLOT + xstages * SH::XF_UNIT + SH::CONV_SLOTS * SH::XF_SLOT)
    return TM_ERR_UNSUPPORTED;
  // the epilogue stages the fp16 tile and s_x of its rows below the barriers
  if (S == 1 && (uint32_t)BT * (256 + 4) > stages * SH::SLOT + xstages * SH::XF_UNIT + SH::CONV_SLOTS * SH::XF_SLOT)
    return TM_ERR_UNSUPPORTED;
  CUtensorMap tmY;
  {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return TM_ERR_CUDA;
    cuuint64_t dims[2] = {(cuuint64_t)p->N, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)p->N * 2};
    cuuint32_t box[2] = {128u, (cuuint32_t)BT};  // 128 output columns x BT rows, 256-byte rows
    cuuint32_t es[2] = {1, 1};
    if (fn(&tmY, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, Y, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return TM_ERR_CUDA;
  }
  CUtensorMap tmX;
  {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return TM_ERR_CUDA;
    cuuint64_t dims[2] = {(cuuint64_t)p->K, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)p->K * (XH ? 2 : 1)};
    cuuint32_t box[2] = {XH ? 64u : 128u, (cuuint32_t)BT};  // 128 bytes per row either way
    cuuint32_t es[2] = {1, 1};
    if (fn(&tmX, XH ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(xq), dims,
           strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return TM_ERR_CUDA;
  }
  W8TcParams P;
  P.sw = p->scales;
  P.sx = sx;
  P.Y = reinterpret_cast<__half*>(Y);
  P.M = M;
  P.N = p->N;
  P.kb_total = p->KB;
  P.kb_per_cta = (p->KB + S - 1) / S;
  P.stages = stages;
  P.xstages = xstages;
  P.x_off = stages * SH::SLOT;
  P.xf_off = P.x_off + xstages * SH::XF_UNIT;
  P.bar_off = P.xf_off + SH::CONV_SLOTS * SH::XF_SLOT;
  return w8tc_launch_t<BT, XH>(tmX, p->tm_codes, tmY, P, dim3((unsigned)MB, (unsigned)NB, (unsigned)S), S, smem,
                               stream);
}

int w8_mt(int M) { return M <= 8 ? 1 : M <= 16 ? 2 : M <= 32 ? 4 : 8; }

// Rows of X per CTA for the tensor-memory kernel: the tile size with the
// smallest estimated time, waves x (rows / relative MMA efficiency) -- an MMA
// of N = 128 costs about as much to issue as its tensor time, so 128-row tiles
// run at roughly 0.55 of the 256-row rate; 64 rows only for M <= 64.
int w8tc_rows(int M, int NT, int sms) {
  if (M <= 64) return 64;
  const int NB = (NT + 7) / 8;
  const double eff[2] = {0.55, 1.0};
  const int rows[2] = {128, 256};
  int best = 128;
  double best_t = 1e30;
  for (int i = 0; i < 2; ++i) {
    const long long tiles = (long long)NB * ((M + rows[i] - 1) / rows[i]);
    const double t = (double)((tiles + sms - 1) / sms) * rows[i] / eff[i];
    if (t < best_t) {
      best_t = t;
      best = rows[i];
    }
  }
  return best;
}

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
  static std::atomic<unsigned long long> attr_done{0};  // one bit per device
  if (!smem_attr_once(attr_done, (const void*)kern, (int)kW8SmemMax)) return TM_ERR_CUDA;
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
  if (cudaLaunchKernelEx(&cfg, w8_quant_act_kernel<false>, reinterpret_cast<const __half*>(X), K, (void*)xq, sx) !=
      cudaSuccess)
    return TM_ERR_CUDA;
  set_launch_count(1);
  return TM_OK;
}

extern "C" tm_status tm_w8a8_quantize_act_f16(const uint16_t* X, int M, int K, uint16_t* xq16, float* sx,
                                              void* stream) {
  if (!X || !xq16 || !sx || M < 0 || K <= 0 || K % 16) return TM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(X) & 15u) || (reinterpret_cast<uintptr_t>(xq16) & 15u) ||
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
  if (cudaLaunchKernelEx(&cfg, w8_quant_act_kernel<true>, reinterpret_cast<const __half*>(X), K, (void*)xq16, sx) !=
      cudaSuccess)
    return TM_ERR_CUDA;
  set_launch_count(1);
  return TM_OK;
}

extern "C" tm_status tm_w8a8_gemm_f16(const uint16_t* xq16, const float* sx, const tm_w8_packed* p, void* Y, int M,
                                      int split_k, int tile_m, void* stream) {
  if (!xq16 || !sx || !p || !Y || M < 0) return TM_ERR_INVALID_ARG;
  if (split_k < 0 || split_k > 8 || (split_k & (split_k - 1))) return TM_ERR_INVALID_ARG;
  if (tile_m != 0 && tile_m != 64 && tile_m != 128 && tile_m != 256) return TM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(xq16) & 15u) || (reinterpret_cast<uintptr_t>(Y) & 15u) ||
      (reinterpret_cast<uintptr_t>(sx) & 3u))
    return TM_ERR_ALIGNMENT;
  if (M == 0) return TM_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int BT = tile_m ? tile_m : w8tc_rows(M, p->NT, num_sms(p->device));
  const tm_status r = BT == 64    ? w8tc_run<64, true>(xq16, sx, p, Y, M, split_k, st)
                      : BT == 128 ? w8tc_run<128, true>(xq16, sx, p, Y, M, split_k, st)
                                  : w8tc_run<256, true>(xq16, sx, p, Y, M, split_k, st);
  if (r == TM_OK) set_launch_count(1);
  return r;
}

extern "C" tm_status tm_w8_quantize_weight(const uint16_t* W, int K, int N, int8_t* q, float* sw, void* stream) {
  if (!W || !q || !sw || K <= 0 || N <= 0 || N % 16) return TM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(W) & 15u) || (reinterpret_cast<uintptr_t>(q) & 7u) ||
      (reinterpret_cast<uintptr_t>(sw) & 3u))
    return TM_ERR_ALIGNMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const dim3 grid((unsigned)((N / 8 + 31) / 32), (unsigned)((K + kWqRows - 1) / kWqRows));
  if (grid.y > 65535u) return TM_ERR_UNSUPPORTED;
  auto* Wh = reinterpret_cast<const __half*>(W);
  auto* amax = reinterpret_cast<uint32_t*>(sw);  // the maxima live in sw until the last launch
  if (cudaMemsetAsync(sw, 0, (size_t)N * 4, st) != cudaSuccess) return TM_ERR_CUDA;
  w8_colmax_kernel<<<grid, 256, 0, st>>>(Wh, K, N, amax);
  w8_wquant_kernel<<<grid, 256, 0, st>>>(Wh, K, N, amax, q);
  w8_scale_kernel<<<(unsigned)((N + 255) / 256), 256, 0, st>>>(sw, N);
  if (cudaGetLastError() != cudaSuccess) return TM_ERR_CUDA;
  set_launch_count(3);
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

extern "C" tm_status tm_w8a8_gemm_ex(const int8_t* xq, const float* sx, const tm_w8_packed* p, void* Y, int M,
                                     int split_k, int tile_m, void* stream) {
  if (!xq || !sx || !p || !Y || M < 0) return TM_ERR_INVALID_ARG;
  if (split_k < 0 || split_k > 8 || (split_k & (split_k - 1))) return TM_ERR_INVALID_ARG;
  if (tile_m != 0 && tile_m != 64 && tile_m != 128 && tile_m != 256) return TM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(xq) & 15u) || (reinterpret_cast<uintptr_t>(Y) & 15u) ||
      (reinterpret_cast<uintptr_t>(sx) & 3u))
    return TM_ERR_ALIGNMENT;
  if (M == 0) return TM_OK;
  if (M > 32) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int BT = tile_m ? tile_m : w8tc_rows(M, p->NT, num_sms(p->device));
    const tm_status r = BT == 64    ? w8tc_run<64, false>(xq, sx, p, Y, M, split_k, st)
                        : BT == 128 ? w8tc_run<128, false>(xq, sx, p, Y, M, split_k, st)
                                    : w8tc_run<256, false>(xq, sx, p, Y, M, split_k, st);
    if (r == TM_OK) set_launch_count(1);
    return r;
  }
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

extern "C" tm_status tm_w8a8_gemm(const int8_t* xq, const float* sx, const tm_w8_packed* p, void* Y, int M,
                                  int split_k, void* stream) {
  return tm_w8a8_gemm_ex(xq, sx, p, Y, M, split_k, 0, stream);
}
