// Decode path (M <= 64): a bandwidth-bound split-K skinny GEMM.
//
// The pages' GEMM pipeline (the guide's diagram, "Pipeline A") streams packed
// weights with cp.async, redistributes them with ldmatrix and dequantises
// with interleaved integer/float work before the MMA.  On sm_103a this kernel
// keeps the idea and changes the machinery:
//   * one elected producer thread streams each CTA's packed codes, scales and
//     zeros into a shared-memory ring with three 1-D bulk async copies
//     (cp.async.bulk) per stage, and the CTA's slice of X with 2-D TMA;
//     consumers wait on mbarriers;
//   * because the packer already stored every 32-bit word in mma.m16n8k16
//     A-fragment order, one 16-byte shared load per lane gives four MMA
//     fragments -- no ldmatrix and no runtime swizzle;
//   * dequantisation: LOP3 mask-and-OR with the 0x6400 (1024.0) pattern turns
//     nibbles into 1024 + q (or 1024 + 16 q); either one HSUB2/HFMA2 per pair
//     gives q - z exactly (9 instructions per 8 weights), or the raw values go
//     straight into the MMA and the zero point and offset are removed once per
//     group with the sum of x (5 instructions per 8 weights plus one product
//     with an all-ones fragment per step, shared by the warp's n-tiles); the
//     fp16 scale multiplies the fp32 per-group partial sum, so no weight is
//     rounded;
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
#include <mutex>

#include "decode_group.h"
#include "tm_common.cuh"

namespace w4 {

constexpr int kGroupMax = TM_GROUP_MAX;  // products of a grouped launch

static __device__ uint32_t s_err_decode;

// One product of a launch.  A launch serves up to G independent products
// with the same M, group size and CTA shape: blockIdx.x runs over the
// clusters of product 0, then those of product 1, and so on.  A cluster of
// C CTAs (C = gridDim.y) holds C / split column blocks of a product, each
// split along K over `split` CTAs; a single-product launch has split == C.
struct DecodeProblem {
  const uint8_t* codes;
  const uint8_t* scales;
  const uint8_t* zeros;
  __half* Y;
  int N, NT;
  int nsg_total;   // pairs of groups
  int sg_per_cta;  // pairs of groups per CTA of a split
  int split;       // CTAs sharing one column block along K (a power of two dividing C)
  int nb;          // clusters (along x) of this product
  int silu;        // Y = silu(gate) * up, [M][N/2] (gate/up interleaved in blocks of 4 columns)
};

template <int G>
struct DecodeParams {
  DecodeProblem prob[G];
  int nprob;
  int M;
  int stages;
  uint32_t x_unit;       // bytes of X per 64-k unit in a stage
  uint32_t x_box;        // bytes one X copy delivers per unit
  uint32_t c_off;        // offset of the codes in a stage
  uint32_t stage_bytes;  // bytes per stage (1024-aligned)
  uint32_t r_off;        // offset of the reduction buffer
  uint32_t bar_off;      // offset of the barriers
};

// X of each product as a 2-D tensor {K, M}.
template <int G>
struct DecodeMaps {
  CUtensorMap x[G];
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

// MT: 8-row tiles of X (M <= 8 MT); WN: n-tiles per consumer warp; NW:
// consumer warps; UPS: 64-k units per stage (2g/64); XP: X stored as M plain
// rows and one zero row (M < 8) instead of 8 MT swizzled rows; G: products
// the launch's tables hold (1, or kGroupMax for a grouped launch).
template <int MT, int WN, int NW, int UPS, bool XP, int G>
__global__ void __launch_bounds__((NW + 1) * 32) decode_kernel(const __grid_constant__ DecodeMaps<G> maps,
                                                               const __grid_constant__ DecodeParams<G> P) {
  constexpr int CN = NW * WN;    // n-tiles per CTA
  constexpr int CNN = CN * 16;   // columns per CTA
  constexpr int UPG = UPS / 2;   // units (of 64 k) per group
  constexpr int NACC = 1;  // accumulator chains per tile (more measured slower)
  // Raw-code products pay off when the all-ones product is shared by several
  // tiles (with one tile per warp they measured slower, single or grouped).
  constexpr bool kRaw = WN >= 2 && MT < 4 * WN;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_base);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // This CTA's product, column block and K slice.
  int cb = blockIdx.x, pi = 0;
  if constexpr (G > 1) {
#pragma unroll
    for (int i = 0; i + 1 < G; ++i)
      if (pi == i && i + 1 < P.nprob && cb >= P.prob[i].nb) {
        cb -= P.prob[i].nb;
        pi = i + 1;
      }
  }
  // Both parameters are __grid_constant__: their fields are read in place
  // where they are used, so nothing of the product stays in registers
  // across the K loop but its index.
  const DecodeProblem& Q = P.prob[pi];
  const CUtensorMap* tmX = &maps.x[pi];
  const int C = gridDim.y;  // CTAs of a cluster
  const int sp = G > 1 ? Q.split : C;
  const int kr = (int)blockIdx.y & (sp - 1);  // rank within the split (the cluster rank is blockIdx.y)
  const int nt0 = (cb * (C / sp) + ((int)blockIdx.y >> (__ffs(sp) - 1))) * CN;
  const int sg_begin = kr * Q.sg_per_cta;
  const int sg_end = min(Q.nsg_total, sg_begin + Q.sg_per_cta);
  const int nsg = nt0 < Q.NT ? max(0, sg_end - sg_begin) : 0;
  const int stages = P.stages;

  const uint32_t bar_full = base + P.bar_off;
  const uint32_t bar_empty = bar_full + 8 * stages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P.bar_off + 16 * stages);
  float* red = reinterpret_cast<float*>(smem + P.r_off);
  const uint32_t s_off = P.c_off + CN * UPS * kUnitBytes;
  const uint32_t z_off = s_off + CN * 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, NW);
    }
    *abort_flag = 0;
    fence_mbar_init();
    launch_dependents();
  }
  if constexpr (XP) {
    // The zero row after the M rows of X in every unit slot: the copies never
    // write it, so it stays zero for the whole kernel.
    for (int i = threadIdx.x; i < stages * UPS * 8; i += blockDim.x) {
      const int s8 = i & 7, su = i >> 3;
      uint8_t* z = smem + (size_t)(su / UPS) * P.stage_bytes + (su % UPS) * P.x_unit + P.M * 128 + s8 * 16;
      *reinterpret_cast<uint4*>(z) = make_uint4(0, 0, 0, 0);
    }
  }
  __syncthreads();
  // Every CTA of the cluster must be running before any CTA stores into its
  // shared memory: arrive now, wait right before the first remote store.
  if (C > 1) cluster_arrive_relaxed();

  if (warp == NW) {
    // ---------------- producer: one elected thread ----------------
    if (lane == 0) {
      prefetch_tmap(tmX);
      const int nvalid = min(CN, Q.NT - nt0);
      const uint32_t tx = UPS * P.x_box + (uint32_t)nvalid * (UPS * kUnitBytes + 64 + 16);
      auto issue_weights = [&](int i) {
        const int slot = i % stages;
        const int sg = sg_begin + i;
        const uint32_t full = bar_full + 8 * slot;
        const uint32_t st = base + slot * P.stage_bytes;
        // one contiguous run each: codes, scales and zeros of n-tiles nt0.. for super-group sg
        const size_t row = (size_t)sg * Q.NT + nt0;
        bulk_g2s(st + P.c_off, Q.codes + row * (UPS * kUnitBytes), (uint32_t)nvalid * UPS * kUnitBytes, full);
        bulk_g2s(st + s_off, Q.scales + row * 64, (uint32_t)nvalid * 64, full);
        bulk_g2s(st + z_off, Q.zeros + row * 16, (uint32_t)nvalid * 16, full);
      };
      auto issue_x = [&](int i) {
        const int slot = i % stages;
        const int sg = sg_begin + i;
        const uint32_t st = base + slot * P.stage_bytes;
#pragma unroll
        for (int u = 0; u < UPS; ++u)
          tma_load_2d(st + u * P.x_unit, tmX, (sg * UPS + u) * kUnitK, 0, bar_full + 8 * slot);
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
    if (C > 1) cluster_wait();
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

    // B fragments of unit u: X rows mt*8 + gr, k = 16t .. 16t+15 (two 16-byte
    // chunks of a 128-byte row).  Plain loads through a generic pointer into
    // shared memory: the compiler may hoist them ahead of earlier MMAs; the
    // barrier wait clobbers memory, so none moves before it.
    auto load_x = [&](const uint8_t* stg, int u, uint4 (&xa)[MT], uint4 (&xb)[MT]) {
      if constexpr (XP) {
        // M plain rows and, after them, a row of zeros that lanes past M read.
        const int r = min(gr, P.M);
        const uint8_t* row = stg + u * P.x_unit + r * 128;
        xa[0] = *reinterpret_cast<const uint4*>(row + 32 * t);
        xb[0] = *reinterpret_cast<const uint4*>(row + 32 * t + 16);
      } else {
        // 8 MT rows, 128-byte swizzle (chunk c of row r at c ^ (r & 7)); rows
        // at or past M were zero-filled by the copy.
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const uint8_t* row = stg + (u * MT + m) * 1024 + gr * 128;
          xa[m] = *reinterpret_cast<const uint4*>(row + (((2 * t) ^ gr) << 4));
          xb[m] = *reinterpret_cast<const uint4*>(row + (((2 * t + 1) ^ gr) << 4));
        }
      }
    };

    int slot = 0;
    uint32_t ph = 0;
    for (int i = 0; i < nsg; ++i) {
      if (!mbar_wait(bar_full + 8 * slot, ph, abort_flag, &s_err_decode)) break;
      const uint8_t* stg = smem + (size_t)slot * P.stage_bytes;
      const uint8_t* cg = stg + P.c_off;
      const uint8_t* sgp = stg + s_off;
      const uint8_t* zg = stg + z_off;
#pragma unroll
      for (int gi = 0; gi < 2; ++gi) {
        float s_lo[WN], s_hi[WN];
        uint32_t zlo[WN], zhi[WN];
#pragma unroll
        for (int j = 0; j < WN; ++j) {
          const int jj = warp * WN + j;
          const uint32_t sp = *reinterpret_cast<const uint32_t*>(sgp + jj * 64 + gi * 32 + gr * 4);
          s_lo[j] = __half2float(__ushort_as_half((unsigned short)(sp & 0xFFFFu)));
          s_hi[j] = __half2float(__ushort_as_half((unsigned short)(sp >> 16)));
          const uint32_t zb = zg[jj * 16 + gi * 8 + gr];
          zlo[j] = zb & 15u;
          zhi[j] = zb >> 4;
        }
        if constexpr (kRaw) {
          // d_lo = sum x (1024 + q), d_hi = sum x (1024 + 16 q) per row pair and
          // xs = sum x (all-ones fragment), so
          // sum x (q - z) = d_lo - (1024 + z) xs = (d_hi - (1024 + 16 z) xs) / 16.
          float zc_lo[WN], zc_hi[WN];
#pragma unroll
          for (int j = 0; j < WN; ++j) {
            zc_lo[j] = (float)(1024u + zlo[j]);
            zc_hi[j] = (float)(1024u + 16u * zhi[j]);
            s_hi[j] *= 0.0625f;
          }
          constexpr uint32_t kOne2 = 0x3C003C00u;  // 1.0 in both halves
          const uint32_t ones[4] = {kOne2, kOne2, kOne2, kOne2};
          float d[WN][MT][4], xs[MT][4];
#pragma unroll
          for (int uu = 0; uu < UPG; ++uu) {
            const int u = gi * UPG + uu;
            uint4 xa[MT], xb[MT];
            load_x(stg, u, xa, xb);
            uint4 cw[WN];
#pragma unroll
            for (int j = 0; j < WN; ++j)
              cw[j] = *reinterpret_cast<const uint4*>(cg + ((warp * WN + j) * UPS + u) * kUnitBytes + lane * 16);
#pragma unroll
            for (int stp = 0; stp < 4; ++stp) {
              const bool first = (uu == 0 && stp == 0);
#pragma unroll
              for (int m = 0; m < MT; ++m) {
                const uint32_t b0 = stp == 0 ? xa[m].x : stp == 1 ? xa[m].z : stp == 2 ? xb[m].x : xb[m].z;
                const uint32_t b1 = stp == 0 ? xa[m].y : stp == 1 ? xa[m].w : stp == 2 ? xb[m].y : xb[m].w;
                if (first) {
                  mma_16816_zc(xs[m], ones, b0, b1);
                } else {
                  mma_16816(xs[m], ones, b0, b1);
                }
              }
#pragma unroll
              for (int j = 0; j < WN; ++j) {
                const uint32_t w = stp == 0 ? cw[j].x : stp == 1 ? cw[j].y : stp == 2 ? cw[j].z : cw[j].w;
                uint32_t a[4];
                raw_word(w, a);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                  const uint32_t b0 = stp == 0 ? xa[m].x : stp == 1 ? xa[m].z : stp == 2 ? xb[m].x : xb[m].z;
                  const uint32_t b1 = stp == 0 ? xa[m].y : stp == 1 ? xa[m].w : stp == 2 ? xb[m].y : xb[m].w;
                  if (first) {
                    mma_16816_zc(d[j][m], a, b0, b1);
                  } else {
                    mma_16816(d[j][m], a, b0, b1);
                  }
                }
              }
            }
          }
#pragma unroll
          for (int j = 0; j < WN; ++j)
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              acc[j][m][0] = fmaf(s_lo[j], fmaf(-zc_lo[j], xs[m][0], d[j][m][0]), acc[j][m][0]);
              acc[j][m][1] = fmaf(s_lo[j], fmaf(-zc_lo[j], xs[m][1], d[j][m][1]), acc[j][m][1]);
              acc[j][m][2] = fmaf(s_hi[j], fmaf(-zc_hi[j], xs[m][0], d[j][m][2]), acc[j][m][2]);
              acc[j][m][3] = fmaf(s_hi[j], fmaf(-zc_hi[j], xs[m][1], d[j][m][3]), acc[j][m][3]);
            }
        } else {
          uint32_t zz[WN], zf[WN];
#pragma unroll
          for (int j = 0; j < WN; ++j) {
            zz[j] = zero_pair_lo(zlo[j]);
            zf[j] = zero_pair_hi(zhi[j]);
          }
          float tmp[NACC][WN][MT][4];
#pragma unroll
          for (int uu = 0; uu < UPG; ++uu) {
            const int u = gi * UPG + uu;
            uint4 xa[MT], xb[MT];
            load_x(stg, u, xa, xb);
            uint4 cw[WN];
#pragma unroll
            for (int j = 0; j < WN; ++j)
              cw[j] = *reinterpret_cast<const uint4*>(cg + ((warp * WN + j) * UPS + u) * kUnitBytes + lane * 16);
#pragma unroll
            for (int stp = 0; stp < 4; ++stp) {
              const int idx = uu * 4 + stp;
              const int c = idx % NACC;
              const bool first = idx < NACC;
#pragma unroll
              for (int j = 0; j < WN; ++j) {
                const uint32_t w = stp == 0 ? cw[j].x : stp == 1 ? cw[j].y : stp == 2 ? cw[j].z : cw[j].w;
                uint32_t a[4];
                dequant_word(w, zz[j], zf[j], a);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                  const uint32_t b0 = stp == 0 ? xa[m].x : stp == 1 ? xa[m].z : stp == 2 ? xb[m].x : xb[m].z;
                  const uint32_t b1 = stp == 0 ? xa[m].y : stp == 1 ? xa[m].w : stp == 2 ? xb[m].y : xb[m].w;
                  if (first) {
                    mma_16816_zc(tmp[c][j][m], a, b0, b1);
                  } else {
                    mma_16816(tmp[c][j][m], a, b0, b1);
                  }
                }
              }
            }
          }
#pragma unroll
          for (int j = 0; j < WN; ++j)
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              float v[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                v[e] = tmp[0][j][m][e];
#pragma unroll
                for (int c = 1; c < NACC; ++c) v[e] += tmp[c][j][m][e];
              }
              acc[j][m][0] = fmaf(s_lo[j], v[0], acc[j][m][0]);
              acc[j][m][1] = fmaf(s_lo[j], v[1], acc[j][m][1]);
              acc[j][m][2] = fmaf(s_hi[j], v[2], acc[j][m][2]);
              acc[j][m][3] = fmaf(s_hi[j], v[3], acc[j][m][3]);
            }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
      if (++slot == stages) {
        slot = 0;
        ph ^= 1u;
      }
    }

    // Partial tile -> the owner of each column slice: red[kr][m][col] in the
    // shared memory of the CTA of this split that owns the slice (its own
    // when the product is not split).
    const int span = CNN / sp;
    const uint32_t owner0 = (uint32_t)(blockIdx.y - kr);  // cluster rank of the split's first CTA
    const uint32_t red_s = smem_u32(red);
    if (C > 1) cluster_wait();
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
          const uint32_t off = (uint32_t)((kr * (MT * 8) + mm) * span + col) * 4u;
          if (sp > 1) {
            st_dsmem_f32(map_shared_rank(red_s + off, owner0 + (uint32_t)owner), acc[j][m][e]);
          } else {
            red[off / 4] = acc[j][m][e];
          }
        }
      }
    }
  }

  // ---------------- reduction of this CTA's column slice ----------------
  if (C > 1) {
    cluster_sync_all();
  } else {
    __syncthreads();
  }
  grid_dependency_wait();  // Y may still be read by the preceding grid
  const int span = CNN / sp;
  const int half_span = span >> 1;
  const int n_base = nt0 * 16 + kr * span;
  if (Q.silu) {
    // Output column j of the slice pairs gate column 8(j/4) + j%4 with the up
    // column 4 later (a slice is a multiple of 8 columns); two outputs a thread.
    const int pairs = span >> 2;
    const int Nh = Q.N >> 1;
    for (int it = threadIdx.x; it < P.M * pairs; it += blockDim.x) {
      const int m = it / pairs;
      const int j = 2 * (it - m * pairs);
      const int c = 8 * (j >> 2) + (j & 3);
      if (n_base + c >= Q.N) continue;
      float2 gt = make_float2(0.f, 0.f), up = make_float2(0.f, 0.f);
#pragma unroll 8
      for (int r = 0; r < sp; ++r) {
        const float* row = red + (r * (MT * 8) + m) * span;
        const float2 a = *reinterpret_cast<const float2*>(row + c);
        const float2 b = *reinterpret_cast<const float2*>(row + c + 4);
        gt.x += a.x;
        gt.y += a.y;
        up.x += b.x;
        up.y += b.y;
      }
      *reinterpret_cast<__half2*>(Q.Y + (size_t)m * Nh + (n_base >> 1) + j) =
          __floats2half2_rn(silu_mul(gt.x, up.x), silu_mul(gt.y, up.y));
    }
    return;
  }
  const int items = P.M * half_span;
  for (int it = threadIdx.x; it < items; it += blockDim.x) {
    const int m = it / half_span;
    const int col = 2 * (it - m * half_span);
    const int n = n_base + col;
    if (n >= Q.N) continue;
    float2 v = make_float2(0.f, 0.f);
#pragma unroll 8
    for (int r = 0; r < sp; ++r) {
      const float2 x = *reinterpret_cast<const float2*>(red + (r * (MT * 8) + m) * span + col);
      v.x += x.x;
      v.y += x.y;
    }
    *reinterpret_cast<__half2*>(Q.Y + (size_t)m * Q.N + n) = __floats2half2_rn(v.x, v.y);
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

constexpr uint32_t kSmemPerCta = 227 * 1024;

int mt_for(int M) { return M <= 8 ? 1 : M <= 16 ? 2 : M <= 32 ? 4 : 8; }

// (tile_n, warp_n) -> (WN n-tiles per warp, NW consumer warps).  Served:
// WN 1 with 4 or 8 warps, WN 2 with 4 or 8 warps (M <= 32), WN 4 with 2 or
// 4 warps (M <= 16).
bool tile_shape(int tile_n, int warp_n, int MT, int* WN, int* NW) {
  if (warp_n != 1 && warp_n != 2 && warp_n != 4) return false;
  if (tile_n % (16 * warp_n)) return false;
  const int nw = tile_n / (16 * warp_n);
  bool ok = false;
  if (warp_n == 1) ok = nw == 4 || nw == 8;
  if (warp_n == 2) ok = (nw == 4 || nw == 8) && MT <= 4;
  if (warp_n == 4) ok = (nw == 2 || nw == 4) && MT <= 2;
  if (!ok) return false;
  *WN = warp_n;
  *NW = nw;
  return true;
}

struct Geometry {
  bool xp;             // X as M plain rows
  uint32_t x_unit;     // bytes of X per unit
  uint32_t c_off;      // codes offset in a stage
  uint32_t stage;      // bytes per stage
  uint32_t red;        // reduction buffer
  uint32_t codes;      // code bytes per stage
};

Geometry geometry(int M, int MT, int CN, int UPS) {
  Geometry g;
  g.xp = MT == 1 && M < 8;
  g.x_unit = g.xp ? (uint32_t)(M + 1) * 128u : (uint32_t)MT * 1024u;  // plain: M rows + a zero row
  g.c_off = UPS * g.x_unit;  // a multiple of 128 (plain) or 1024 (swizzled)
  g.codes = (uint32_t)CN * UPS * kUnitBytes;
  g.stage = (g.c_off + g.codes + CN * 80u + 1023u) & ~1023u;
  g.red = (uint32_t)MT * 8 * CN * 16 * 4;
  return g;
}

uint32_t smem_bytes(const Geometry& g, int stages) {
  const uint32_t bar_off = (g.stage * stages + g.red + 15u) & ~15u;
  return bar_off + 16 * stages + 16 + 1024;  // + alignment slack
}

// Largest stage count that fits `budget` bytes of shared memory.
int fit_stages(const Geometry& g, uint32_t budget) {
  int s = 8;
  while (s >= 2 && smem_bytes(g, s) > budget) --s;
  return s;
}

// Shared memory to request per CTA so that at most ceil(ctas / SMs) CTAs of
// the launch fit on one SM.  Measured on GB300 over the Llama-3 8B/70B decode
// shapes: when more CTAs fit than the even share, the block scheduler packs
// clusters onto fewer SMs and the launch runs up to 1.5x slower; capping
// residency at the even share keeps every SM's copy engine streaming.  The
// padding is also the budget for ring stages.
uint32_t residency_budget(int device, int ctas) {
  int per_sm = 0, reserved = 0;
  sm_shared_memory(device, &per_sm, &reserved);
  const int sms = num_sms(device);
  const int r = std::max(1, (ctas + sms - 1) / sms);
  const int b = per_sm / r - reserved;
  return (uint32_t)std::min<int>((int)kSmemPerCta, std::max(0, b)) & ~127u;
}

// With `query` set, returns the kernel through it instead of launching.
template <int MT, int WN, int NW, int UPS, bool XP, int G>
tm_status launch_t(const DecodeMaps<G>& maps, const DecodeParams<G>& P, int blocks, int C, uint32_t smem,
                   cudaStream_t stream, const void** query) {
  auto kern = decode_kernel<MT, WN, NW, UPS, XP, G>;
  if (query) {
    *query = (const void*)kern;
    return TM_OK;
  }
  static std::atomic<unsigned long long> attr_done{0};  // per instantiation, one bit per device
  if (!smem_attr_once(attr_done, (const void*)kern, (int)kSmemPerCta)) return TM_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, (unsigned)C, 1);
  cfg.blockDim = dim3((NW + 1) * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  int na = 0;
  at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (C > 1) {
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = 1;
    at[na].val.clusterDim.y = (unsigned)C;
    at[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, maps, P);
  return e == cudaSuccess ? TM_OK : TM_ERR_CUDA;
}

template <int MT, int WN, int NW, bool XP, int G>
tm_status launch_u(int UPS, const DecodeMaps<G>& maps, const DecodeParams<G>& P, int blocks, int C, uint32_t smem,
                   cudaStream_t stream, const void** query) {
  return UPS == 4 ? launch_t<MT, WN, NW, 4, XP, G>(maps, P, blocks, C, smem, stream, query)
                  : launch_t<MT, WN, NW, 2, XP, G>(maps, P, blocks, C, smem, stream, query);
}

// Served CTA shapes: WN 1 with 4 or 8 warps; for a single product also WN 2
// with 4 or 8 warps (M <= 32) and WN 4 with 2 or 4 warps (M <= 16).  (Two
// tiles a warp in a grouped launch measured slower: 32.3 against 26.8 us
// for the 8B layer at M = 1.)
template <int MT, bool XP, int G>
tm_status launch_m(int WN, int NW, int UPS, const DecodeMaps<G>& maps, const DecodeParams<G>& P, int blocks, int C,
                   uint32_t smem, cudaStream_t stream, const void** query) {
  if (WN == 1 && NW == 4) return launch_u<MT, 1, 4, XP, G>(UPS, maps, P, blocks, C, smem, stream, query);
  if (WN == 1 && NW == 8) return launch_u<MT, 1, 8, XP, G>(UPS, maps, P, blocks, C, smem, stream, query);
  if constexpr (MT <= 4 && G == 1) {
    if (WN == 2 && NW == 4) return launch_u<MT, 2, 4, XP, G>(UPS, maps, P, blocks, C, smem, stream, query);
    if (WN == 2 && NW == 8) return launch_u<MT, 2, 8, XP, G>(UPS, maps, P, blocks, C, smem, stream, query);
  }
  if constexpr (MT <= 2 && G == 1) {
    if (WN == 4 && NW == 2) return launch_u<MT, 4, 2, XP, G>(UPS, maps, P, blocks, C, smem, stream, query);
    if (WN == 4 && NW == 4) return launch_u<MT, 4, 4, XP, G>(UPS, maps, P, blocks, C, smem, stream, query);
  }
  return TM_ERR_UNSUPPORTED;
}

// Launch (or, with `query`, look up) the instantiation for MT, XP, WN, NW, UPS.
template <int G>
tm_status dispatch(int MT, bool XP, int WN, int NW, int UPS, const DecodeMaps<G>& maps, const DecodeParams<G>& P,
                   int blocks, int C, uint32_t smem, cudaStream_t stream, const void** query) {
  switch (MT) {
    case 1:
      return XP ? launch_m<1, true, G>(WN, NW, UPS, maps, P, blocks, C, smem, stream, query)
                : launch_m<1, false, G>(WN, NW, UPS, maps, P, blocks, C, smem, stream, query);
    case 2: return launch_m<2, false, G>(WN, NW, UPS, maps, P, blocks, C, smem, stream, query);
    case 4: return launch_m<4, false, G>(WN, NW, UPS, maps, P, blocks, C, smem, stream, query);
    case 8: return launch_m<8, false, G>(WN, NW, UPS, maps, P, blocks, C, smem, stream, query);
    default: return TM_ERR_UNSUPPORTED;
  }
}

// Resident CTAs per SM that the registers and threads of the grouped
// instantiation allow (occupancy calculator at a small shared-memory
// request), cached per instantiation.
int group_ctas_by_registers(int MT, bool XP, int WN, int NW, int UPS) {
  static std::mutex mu;
  static int cache[4][2][2][2][2] = {};  // MT index, XP, WN 1/2, NW 4/8, UPS 2/4
  const int mi = MT == 1 ? 0 : MT == 2 ? 1 : MT == 4 ? 2 : 3;
  std::lock_guard<std::mutex> lk(mu);
  int& c = cache[mi][XP ? 1 : 0][WN == 2 ? 1 : 0][NW == 8 ? 1 : 0][UPS == 4 ? 1 : 0];
  if (c) return c;
  const void* k = nullptr;
  const DecodeMaps<kGroupMax> maps = {};
  const DecodeParams<kGroupMax> P = {};
  if (dispatch<kGroupMax>(MT, XP, WN, NW, UPS, maps, P, 1, 1, 0, nullptr, &k) != TM_OK || !k) return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, (NW + 1) * 32, 4096) != cudaSuccess || n < 1) n = 1;
  c = n;
  return c;
}

}  // namespace

// Launch shape.  Measured on GB300 over the Llama-3 8B/70B decode shapes:
// 128 columns per CTA (64 for short K with few columns; else the other,
// else 256) and the smallest cluster split giving at least 256 CTAs; shared
// memory padded so that each SM holds an even share of the CTAs
// (residency_budget), and as many ring stages as that budget holds, up to
// the CTA's super-group count.
tm_status plan_decode(const tm_packed* p, int M, const tm_gemm_config* in, tm_gemm_config* out) {
  const Layout& L = p->L;
  const int MT = mt_for(M);
  const int want_tile = in ? in->tile_n : 0;
  const int want_S = in ? in->split_k : 0;
  const int want_stages = in ? in->stages : 0;
  const int want_wn = in ? in->warp_n : 0;
  if (want_tile && want_tile != 64 && want_tile != 128 && want_tile != 256) return TM_ERR_INVALID_ARG;
  if (want_S && want_S != 1 && want_S != 2 && want_S != 4 && want_S != 8) return TM_ERR_INVALID_ARG;
  if (want_stages && (want_stages < 2 || want_stages > 8)) return TM_ERR_INVALID_ARG;
  if (want_wn && want_wn != 1 && want_wn != 2 && want_wn != 4) return TM_ERR_INVALID_ARG;
  constexpr int kMinCtas = 256;
  // 128 columns per CTA first, unless that needs a cluster of 8 CTAs that
  // each hold fewer than 4 super-groups of K: then 64 columns (half the
  // cluster, the same CTA count) measured faster.
  const bool narrow = (L.NT + 7) / 8 * 4 < kMinCtas && L.NSG < 32;
  const int tiles[3] = {narrow ? 64 : 128, narrow ? 128 : 64, 256};
  const int splits[4] = {1, 2, 4, 8};
  tm_gemm_config pick = {0, 0, 0, 0, 0, 0};
  tm_gemm_config fallback = {0, 0, 0, 0, 0, 0};  // the shape with the most CTAs
  int fallback_ctas = 0;
  for (int tile : tiles) {
    if (want_tile && tile != want_tile) continue;
    // one 16-column tile per warp unless requested otherwise (measured fastest);
    // a tile only served with more per warp takes the first that fits
    int WN = 0, NW = 0, wn = 0;
    const int wns[3] = {1, 2, 4};
    for (int w : wns) {
      if (want_wn && w != want_wn) continue;
      if (tile_shape(tile, w, MT, &WN, &NW)) {
        wn = w;
        break;
      }
    }
    if (!wn) continue;
    const int CN = WN * NW;
    const int NB = (L.NT + CN - 1) / CN;
    const Geometry g = geometry(M, MT, CN, L.UPS);
    for (int S : splits) {
      if (want_S && S != want_S) continue;
      if (!want_S && S > 1 && S > L.NSG) break;
      const int per_cta = (L.NSG + S - 1) / S;
      const uint32_t budget = residency_budget(p->device, NB * S);
      int stages = want_stages ? want_stages : std::min(std::max(2, per_cta), std::max(2, fit_stages(g, budget)));
      if (stages < 2 || smem_bytes(g, stages) > kSmemPerCta) continue;
      const tm_gemm_config c = {1, S, tile, stages, wn, 0};
      if (NB * S > fallback_ctas) {
        fallback = c;
        fallback_ctas = NB * S;
      }
      if (NB * S >= kMinCtas || want_S) {
        pick = c;
        break;
      }
    }
    if (pick.path) break;
  }
  if (pick.path == 0) pick = fallback;
  if (pick.path == 0) return TM_ERR_UNSUPPORTED;
  *out = pick;
  return TM_OK;
}


namespace {

// X as a 2-D tensor {K, M}: box = 64 k x rows; rows beyond M and columns
// beyond K read as zeros.  8 MT rows with a 128-byte swizzle, or exactly M
// plain rows when M < 8.
bool encode_x(CUtensorMap* m, const void* X, int K, int M, int MT, bool xp) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)(xp ? M : 8 * MT)};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(X), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, xp ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One launch over n products that share M and the group size: the launch
// settings c (c.split_k = C, the cluster size) and each product's split
// (a power of two dividing C).  A single product pads shared memory to the
// even share of the resident CTAs (residency_budget); a grouped launch runs
// several waves and takes the stage count c gives.
template <int G>
tm_status launch_group(const DecodeJob* jobs, const int* splits, int n, int M, const tm_gemm_config& c,
                       cudaStream_t stream) {
  if (n < 1 || n > G) return TM_ERR_INVALID_ARG;
  const Layout& L0 = jobs[0].p->L;
  const int MT = mt_for(M);
  int WN = 0, NW = 0;
  if (!tile_shape(c.tile_n, c.warp_n, MT, &WN, &NW)) return TM_ERR_UNSUPPORTED;
  const int CN = WN * NW;
  const int C = c.split_k;
  const Geometry g = geometry(M, MT, CN, L0.UPS);
  DecodeMaps<G> maps = {};
  DecodeParams<G> P = {};
  int blocks = 0;
  for (int i = 0; i < n; ++i) {
    const Layout& L = jobs[i].p->L;
    const int sp = splits[i];
    if (L.UPS != L0.UPS || sp < 1 || sp > C || C % sp != 0 || (sp & (sp - 1))) return TM_ERR_INVALID_ARG;
    if (!encode_x(&maps.x[i], jobs[i].X, L.K, M, MT, g.xp)) return TM_ERR_CUDA;
    DecodeProblem& Q = P.prob[i];
    Q.codes = jobs[i].p->base + L.codes_off;
    Q.scales = jobs[i].p->base + L.scales_off;
    Q.zeros = jobs[i].p->base + L.zeros_off;
    Q.Y = reinterpret_cast<__half*>(jobs[i].Y);
    Q.N = L.N;
    Q.NT = L.NT;
    Q.nsg_total = L.NSG;
    Q.split = sp;
    Q.sg_per_cta = (L.NSG + sp - 1) / sp;
    const int per_cluster = C / sp;  // column blocks a cluster holds
    Q.nb = ((L.NT + CN - 1) / CN + per_cluster - 1) / per_cluster;
    Q.silu = jobs[i].silu ? 1 : 0;
    blocks += Q.nb;
  }
  P.nprob = n;
  P.M = M;
  P.stages = c.stages;
  P.x_unit = g.x_unit;
  P.x_box = g.xp ? (uint32_t)M * 128u : (uint32_t)MT * 1024u;
  P.c_off = g.c_off;
  P.stage_bytes = g.stage;
  P.r_off = g.stage * c.stages;
  P.bar_off = (P.r_off + g.red + 15u) & ~15u;
  const uint32_t need = smem_bytes(g, c.stages);
  if (need > kSmemPerCta) return TM_ERR_UNSUPPORTED;
  const uint32_t smem = G == 1 ? std::max(need, residency_budget(jobs[0].p->device, blocks * C)) : need;
  const tm_status st = dispatch<G>(MT, g.xp, WN, NW, L0.UPS, maps, P, blocks, C, smem, stream, nullptr);
  if (st == TM_OK) set_launch_count(1);
  return st;
}

// Split of one product of an automatic grouped launch: 2, doubled (up to
// 8) while its K slice would exceed 8192 rows of W.  Measured on the Llama-3
// 8B decode layers (M = 1..32, 64-column CTAs): a split of 2 for every
// product beat 1 (the longest slices then set the launch time), 4, and
// splits equalising the slices ([2, 2, 2, 8]): more CTAs add start-ups and
// reductions that the weight stream does not hide.
int group_auto_split(const Layout& L) {
  const int cap = std::max(1, 8192 / (2 * L.g));  // super-groups
  int sp = 2;
  while (sp < 8 && (L.NSG + sp - 1) / sp > cap) sp *= 2;
  return sp;
}

}  // namespace

tm_status launch_decode(const void* X, const tm_packed* p, void* Y, int M, const tm_gemm_config& c,
                        cudaStream_t stream, bool silu) {
  const DecodeJob job = {X, p, Y, silu};
  const int split = c.split_k;
  return launch_group<1>(&job, &split, 1, M, c, stream);
}

// Launch settings of a grouped launch: one CTA shape and one cluster size
// for every product, a split per product.  Automatic: 64-column CTAs of four
// warps; each product's split by group_auto_split, the cluster the largest
// of them; stages for the even share of the resident CTAs (at most the
// registers' limit per SM), up to the longest slice -- in practice two:
// deeper rings measured slower, as they leave fewer CTAs on an SM -- but
// no more than 8 CTAs an SM.  An explicit split_k splits every product that
// many ways.
tm_status plan_decode_group(const tm_packed* const* ps, int n, int M, const tm_gemm_config* in, tm_gemm_config* out,
                            int* splits) {
  if (n < 1 || n > kGroupMax) return TM_ERR_INVALID_ARG;
  const int MT = mt_for(M);
  const int want_tile = in ? in->tile_n : 0;
  const int want_S = in ? in->split_k : 0;
  const int want_stages = in ? in->stages : 0;
  const int want_wn = in ? in->warp_n : 0;
  if (want_tile && want_tile != 64 && want_tile != 128) return TM_ERR_UNSUPPORTED;
  if (want_S && want_S != 1 && want_S != 2 && want_S != 4 && want_S != 8) return TM_ERR_INVALID_ARG;
  if (want_stages && (want_stages < 2 || want_stages > 8)) return TM_ERR_INVALID_ARG;
  if (want_wn && want_wn != 1) return TM_ERR_UNSUPPORTED;
  const int tile = want_tile ? want_tile : 64;
  const int wn = 1;
  int WN = 0, NW = 0;
  if (!tile_shape(tile, wn, MT, &WN, &NW)) return TM_ERR_UNSUPPORTED;
  const int CN = WN * NW;
  int sp[kGroupMax];
  int C = 1;
  for (int i = 0; i < n; ++i) {
    if (!ps[i] || ps[i]->L.UPS != ps[0]->L.UPS) return TM_ERR_INVALID_ARG;
    sp[i] = want_S ? want_S : group_auto_split(ps[i]->L);
    C = std::max(C, sp[i]);
  }
  int ctas = 0, per_cta = 0;
  for (int i = 0; i < n; ++i) {
    const int per_cluster = C / sp[i];
    ctas += ((ps[i]->L.NT + CN - 1) / CN + per_cluster - 1) / per_cluster * C;
    per_cta = std::max(per_cta, (ps[i]->L.NSG + sp[i] - 1) / sp[i]);
  }
  const Geometry g = geometry(M, MT, CN, ps[0]->L.UPS);
  int stages = want_stages;
  if (!stages) {
    int per_sm = 0, reserved = 0;
    sm_shared_memory(ps[0]->device, &per_sm, &reserved);
    const int sms = num_sms(ps[0]->device);
    const int r = std::max(1, std::min((ctas + sms - 1) / sms, group_ctas_by_registers(MT, g.xp, WN, NW, ps[0]->L.UPS)));
    const uint32_t budget = std::min<uint32_t>((uint32_t)std::max(0, per_sm / r - reserved), kSmemPerCta);
    stages = std::min(std::max(2, per_cta), std::max(2, fit_stages(g, budget)));
    // At most 8 CTAs an SM: a 1-row launch with 2 stages fits 9, and when a
    // launch of another M follows it under programmatic dependent launch,
    // that launch's larger CTAs take the slots unevenly (the Llama-3 8B
    // decode step, M = 1 then 8: 38 against 29 us per launch); 3 stages
    // measured faster for M = 1 on its own as well.
    while (stages < 8 && stages < per_cta &&
           per_sm / (int)(smem_bytes(g, stages) + reserved) > 8 && smem_bytes(g, stages + 1) <= kSmemPerCta)
      ++stages;
  }
  if (smem_bytes(g, stages) > kSmemPerCta) return TM_ERR_UNSUPPORTED;
  *out = {1, C, tile, stages, wn, 0};
  if (splits)
    for (int i = 0; i < n; ++i) splits[i] = sp[i];
  return TM_OK;
}

tm_status launch_decode_group(const DecodeJob* jobs, int n, int M, const tm_gemm_config* in, cudaStream_t stream) {
  if (n < 1 || n > kGroupMax) return TM_ERR_INVALID_ARG;
  const tm_packed* ps[kGroupMax];
  for (int i = 0; i < n; ++i) ps[i] = jobs[i].p;
  tm_gemm_config c;
  int splits[kGroupMax];
  tm_status st = plan_decode_group(ps, n, M, in, &c, splits);
  if (st != TM_OK) return st;
  // Longest K slice first, so that the long CTAs start in the first wave.
  int order[kGroupMax];
  for (int i = 0; i < n; ++i) order[i] = i;
  std::stable_sort(order, order + n, [&](int a, int b) {
    return (ps[a]->L.NSG + splits[a] - 1) / splits[a] > (ps[b]->L.NSG + splits[b] - 1) / splits[b];
  });
  DecodeJob sorted[kGroupMax];
  int sorted_splits[kGroupMax];
  for (int i = 0; i < n; ++i) {
    sorted[i] = jobs[order[i]];
    sorted_splits[i] = splits[order[i]];
  }
  return launch_group<kGroupMax>(sorted, sorted_splits, n, M, c, stream);
}

}  // namespace w4
