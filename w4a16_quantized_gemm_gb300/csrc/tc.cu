// Tensor-memory path: Y = X . dequant(W) on tcgen05 with W^T as the A operand
// in tensor memory (TMEM) and X as the B operand in shared memory.
//
// The pages' pipeline (the guide's diagram, "Pipeline A") stages dequantised
// weights in shared memory for the tensor cores.  On sm_103a that staging is
// the bottleneck: every dequantised tile is written to shared memory and read
// back by the tensor core, on top of the X tile, and shared-memory bandwidth
// runs out long before the tensor pipe.  tcgen05.mma can take its A operand
// from tensor memory instead, so here the dequantising warps write W^T
// straight into TMEM (tcgen05.st) and shared memory carries only the TMA
// traffic (X, codes, scales, zeros):
//   * warp 0, one thread: TMA per 64-k block into a ring -- the packed codes
//     of 8 n-tiles (as 128-byte rows with the 128-byte swizzle), their scales
//     and zeros, and the X tile (BT rows x 64 k, 128-byte swizzle).  The
//     weights of the first ring slots are requested before the preceding
//     kernel in the stream has finished (programmatic dependent launch); X
//     waits for it;
//   * warps 2..9: one n-tile each.  A lane reads its four code words
//     transposed across the lanes of its quad (four conflict-free 32-bit
//     shared loads thanks to the swizzle), so that word s holds rows gr,
//     gr + 8 at k = 16s + 4t .. +3; (q - z) exactly in fp16, times s rounded
//     once to fp16, and tcgen05.st.16x256b puts the pairs where the MMA's A
//     operand expects them (lane = output column, column c = k pair c);
//   * warp 1, one thread: tcgen05.mma kind::f16, M = 128 (output columns),
//     N = BT (rows of X), K = 16, fp32 accumulators in TMEM; commits free the
//     ring slot and the TMEM A slot;
//   * warps 2..9 again: epilogue TMEM -> registers -> fp16 -> Y.
// Small problems split K over a cluster of S CTAs and reduce the fp32 tiles
// through distributed shared memory (reusing the ring), in rank order.
// All waits are bounded; a timeout raises a device error bit and the CTA
// unwinds without leaving copies or MMAs in flight.
#include <algorithm>

#include "tm_common.cuh"

namespace w4 {

static __device__ uint32_t s_err_tc;

constexpr int kTcThreads = 320;  // 10 warps
constexpr int kTcTiles = 8;      // n-tiles per CTA: 128 output columns = the MMA's M
constexpr int kTcUnit = 64;      // k per packed unit

// BT rows of X per CTA, KU 64-k units per ring slot, SB tensor-memory A slots.
template <int BT, int KU, int SB>
struct TcShape {
  static constexpr uint32_t C_UNIT = kTcTiles * kUnitBytes;  // 4 KB of codes per unit
  static constexpr uint32_t X_UNIT = BT * kTcUnit * 2;       // BT rows x 64 k fp16 per unit
  static constexpr uint32_t C_OFF = 0;
  static constexpr uint32_t X_OFF = KU * C_UNIT;
  static constexpr uint32_t S_OFF = X_OFF + KU * X_UNIT;  // both groups of the super-group
  static constexpr uint32_t Z_OFF = S_OFF + 2 * kTcTiles * 32;
  static constexpr uint32_t SLOT = (Z_OFF + kTcTiles * 16 + 1023) & ~1023u;
  static constexpr uint32_t TX = KU * (C_UNIT + X_UNIT) + 2 * kTcTiles * 32 + kTcTiles * 16;
  static constexpr uint32_t A_COLS = KU * 32;  // 8 columns per 16 k
  static constexpr uint32_t TMEM_COLS = BT + SB * A_COLS <= 256 ? 256 : 512;
  static constexpr uint32_t A_COL = TMEM_COLS - SB * A_COLS;  // first A slot column
  static_assert(BT + SB * A_COLS <= 512, "tensor memory holds 512 columns");
  static_assert(X_OFF % 1024 == 0 && X_UNIT % 1024 == 0, "swizzled tiles need 1024-byte alignment");
};

struct TcParams {
  __half* Y;
  int M, N, NT, UPS, g;
  int kb_total;    // 64-k units
  int kb_per_cta;  // 64-k units per CTA of a cluster (a multiple of KU)
  int stages;      // ring slots
  uint32_t bar_off;
  int silu;        // Y = silu(gate) * up, [M][N/2] (gate/up interleaved in blocks of 4 columns)
};

__device__ __forceinline__ bool tc_wait_time_only(uint32_t bar, uint32_t parity) {
  unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) {
      atomicOr(&s_err_tc, kErrTimeout);
      return false;
    }
  }
  return true;
}

template <int BT, int KU, int SB>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmC,
              const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmZ,
              const __grid_constant__ CUtensorMap tmY, const TcParams P) {
  using SH = TcShape<BT, KU, SB>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_base);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt0 = blockIdx.x * kTcTiles;
  const int m0 = blockIdx.y * BT;
  const int S = gridDim.z;
  const int kb0 = blockIdx.z * P.kb_per_cta;
  const int nkb = max(0, min(P.kb_total, kb0 + P.kb_per_cta) - kb0);
  const int nst = nkb / KU;  // ring rounds (kb_per_cta and kb_total are multiples of KU)
  const int SA = P.stages;

  const uint32_t barA = base + P.bar_off;  // [SA] full, then [SA] empty
  const uint32_t barT = barA + 16 * SA;    // [SB] full, then [SB] empty (TMEM A slots)
  const uint32_t bar_acc = barT + 16 * SB;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + P.bar_off + 16 * SA + 16 * SB + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P.bar_off + 16 * SA + 16 * SB + 12);
  auto fullA = [&](int s) { return barA + 8 * s; };
  auto emptyA = [&](int s) { return barA + 8 * (SA + s); };
  auto fullT = [&](int s) { return barT + 8 * s; };
  auto emptyT = [&](int s) { return barT + 8 * (SB + s); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < SA; ++s) {
      mbar_init(fullA(s), 1);
      mbar_init(emptyA(s), 1);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(fullT(s), kTcTiles);
      mbar_init(emptyT(s), 1);
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
      prefetch_tmap(&tmC);
      prefetch_tmap(&tmS);
      prefetch_tmap(&tmZ);
      auto issue_w = [&](int i, int s) {
        const int kb = kb0 + i * KU;
        const int sg = kb / P.UPS, u0 = kb - sg * P.UPS;
        const uint32_t st = base + s * SH::SLOT;
#pragma unroll
        for (int u = 0; u < KU; ++u) tma_load_5d(st + SH::C_OFF + u * SH::C_UNIT, &tmC, 0, 0, u0 + u, nt0, sg, fullA(s));
        tma_load_4d(st + SH::S_OFF, &tmS, 0, 0, nt0, sg, fullA(s));
        tma_load_4d(st + SH::S_OFF + kTcTiles * 32, &tmS, 0, 1, nt0, sg, fullA(s));
        tma_load_3d(st + SH::Z_OFF, &tmZ, 0, nt0, sg, fullA(s));
      };
      auto issue_x = [&](int i, int s) {
        const int kb = kb0 + i * KU;
        const uint32_t st = base + s * SH::SLOT + SH::X_OFF;
#pragma unroll
        for (int u = 0; u < KU; ++u) tma_load_2d(st + u * SH::X_UNIT, &tmX, (kb + u) * kTcUnit, m0, fullA(s));
      };
      // Weights first: they do not depend on the preceding kernel; X does.
      const int first = min(nst, SA);
      for (int i = 0; i < first; ++i) {
        mbar_expect_tx(fullA(i), SH::TX);
        issue_w(i, i);
      }
      grid_dependency_wait();
      for (int i = 0; i < first; ++i) issue_x(i, i);
      int issued = first;
      int s = first % SA;
      uint32_t ph = first == SA ? 1u : 0u;
      for (int i = first; i < nst; ++i) {
        if (!mbar_wait(emptyA(s), ph ^ 1u, abort_flag, &s_err_tc)) break;
        mbar_expect_tx(fullA(s), SH::TX);
        issue_w(i, s);
        issue_x(i, s);
        ++issued;
        if (++s == SA) {
          s = 0;
          ph ^= 1u;
        }
      }
      // Never leave with copies in flight into this CTA's shared memory.
      for (int i = max(0, issued - SA); i < issued; ++i) tc_wait_time_only(fullA(i % SA), (uint32_t)(i / SA) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(128, BT);
      int sa = 0, sb = 0;
      uint32_t pa = 0, pb = 0;
      for (int i = 0; i < nst; ++i) {
        if (!mbar_wait(fullA(sa), pa, abort_flag, &s_err_tc)) break;
        if (!mbar_wait(fullT(sb), pb, abort_flag, &s_err_tc)) break;
        tc_fence_after();
        const uint64_t db = smem_desc_sw128(base + sa * SH::SLOT + SH::X_OFF);
        const uint32_t ta = tmem + SH::A_COL + SH::A_COLS * sb;
#pragma unroll
        for (int u = 0; u < KU; ++u)
#pragma unroll
          for (int k = 0; k < kTcUnit / 16; ++k)
            tc_mma_f16_ta(tmem, ta + 8u * (4 * u + k), db + (uint64_t)((u * SH::X_UNIT) >> 4) + (uint64_t)(2 * k),
                          idesc, (i > 0 || u > 0 || k > 0) ? 1u : 0u);
        tc_commit(emptyA(sa));
        tc_commit(emptyT(sb));
        if (++sa == SA) {
          sa = 0;
          pa ^= 1u;
        }
        if (++sb == SB) {
          sb = 0;
          pb ^= 1u;
        }
      }
      // Completes once every MMA issued above has finished (also on abort).
      tc_commit(bar_acc);
    }
    __syncwarp();
  } else {
    // ---------------- dequantisers: one n-tile per warp ----------------
    const int q = warp & 3;         // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;  // which of the quarter's two n-tiles
    const int j = 2 * q + h;        // n-tile within the CTA
    const uint32_t lane_off = (uint32_t)(32 * q + 16 * h) << 16;
    const int gr = lane >> 2, t = lane & 3;
    // Word t of lanes 4 gr + s (s = 0..3): a unit of one n-tile is 4 rows of
    // 128 bytes, 16-byte chunk c of row r stored at c ^ (r & 7).
    const int crow = 4 * j + (gr >> 1);
    uint32_t coff[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) coff[s] = crow * 128 + ((((4 * (gr & 1) + s) ^ (crow & 7))) << 4) + 4 * t;
    const int units_per_group = P.g / kTcUnit;
    int sa = 0, sb = 0;
    uint32_t pa = 0, pb = 0;
    for (int i = 0; i < nst; ++i) {
      if (!mbar_wait(fullA(sa), pa, abort_flag, &s_err_tc)) break;
      if (!mbar_wait(emptyT(sb), pb ^ 1u, abort_flag, &s_err_tc)) break;
      tc_fence_after();
      const uint32_t st = base + sa * SH::SLOT;
      const int u0 = (kb0 + i * KU) % P.UPS;  // first unit of the slot within its super-group
      // All shared loads of the slot first, so that their latencies overlap.
      uint32_t w[KU][4], sp[KU];
#pragma unroll
      for (int u = 0; u < KU; ++u) {
#pragma unroll
        for (int s = 0; s < 4; ++s) w[u][s] = lds32(st + SH::C_OFF + u * SH::C_UNIT + coff[s]);
        const int gi = (u0 + u) / units_per_group;  // group within the super-group
        sp[u] = lds32(st + SH::S_OFF + gi * (kTcTiles * 32) + j * 32 + gr * 4);
      }
      const uint32_t zw0 = lds32(st + SH::Z_OFF + j * 16 + (gr & ~3));
      const uint32_t zw1 = lds32(st + SH::Z_OFF + j * 16 + 8 + (gr & ~3));
      const uint32_t ta = tmem + lane_off + SH::A_COL + SH::A_COLS * sb;
#pragma unroll
      for (int u = 0; u < KU; ++u) {
        const int gi = (u0 + u) / units_per_group;
        const uint32_t zb = ((gi ? zw1 : zw0) >> (8 * (gr & 3))) & 0xFFu;
        const uint32_t zz = zero_pair_lo(zb & 15u), zf = zero_pair_hi(zb >> 4);
        const uint32_t s_lo = (sp[u] & 0xFFFFu) | (sp[u] << 16);      // s of row gr, twice
        const uint32_t s_hi = (sp[u] >> 16) | (sp[u] & 0xFFFF0000u);  // s of row gr+8, twice
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          uint32_t o[4];
          dequant_word(w[u][s], zz, zf, o);
          // lane gr: k 4t, 4t+1 | 4t+2, 4t+3 of slice 4u + s; lane gr + 8 likewise
          tc_st_16x256b(ta + 8u * (4 * u + s), hmul2_u32(o[0], s_lo), hmul2_u32(o[2], s_lo),
                        hmul2_u32(o[1], s_hi), hmul2_u32(o[3], s_hi));
        }
      }
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(fullT(sb));
      if (++sa == SA) {
        sa = 0;
        pa ^= 1u;
      }
      if (++sb == SB) {
        sb = 0;
        pb ^= 1u;
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
  if (epi) {
    acc_ok = mbar_wait(bar_acc, 0, abort_flag, &s_err_tc);
    acc_ok = __all_sync(0xffffffffu, acc_ok);  // warp-uniform: the epilogue shuffles
    tc_fence_after();
  }
  if (S == 1 && P.silu) {
    if (epi) grid_dependency_wait();  // Y may still be read by the preceding grid
    if (epi && acc_ok) {
      const int n = nt0 * 16 + row;
#pragma unroll 1
      for (int c = 0; c < HALF; c += 8) {
        uint32_t v[8];
        tc_ld_32x32b_x8(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(h * HALF + c), v);
        tc_wait_ld();
        if (P.silu) {
          // lanes with (n & 4) == 0 hold gate columns; their up columns sit 4 lanes higher
          float up[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) up[e] = __shfl_down_sync(0xffffffffu, __uint_as_float(v[e]), 4);
          if (n < P.N && (n & 4) == 0) {
            const int j = 4 * (n >> 3) + (n & 3);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int m = m0 + h * HALF + c + e;
              if (m < P.M) P.Y[(size_t)m * (P.N >> 1) + j] = __float2half_rn(silu_mul(__uint_as_float(v[e]), up[e]));
            }
          }
        } else if (n < P.N) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int m = m0 + h * HALF + c + e;
            if (m < P.M) P.Y[(size_t)m * P.N + n] = __float2half_rn(__uint_as_float(v[e]));
          }
        }
      }
    }
  } else if (S == 1) {
    // The ring is idle once the accumulator is complete (every copy was
    // consumed by an MMA): the fp16 tile is staged there, rows of 128
    // columns (256 bytes), and leaves in one TMA tensor store that clips rows
    // past M and columns past N.
    constexpr int CH = HALF < 32 ? HALF : 32;  // accumulator columns per TMEM wait
    const uint32_t ystage = base;
    if (epi && acc_ok) {
#pragma unroll 1
      for (int c = 0; c < HALF; c += CH) {
        uint32_t v[CH];
#pragma unroll
        for (int b = 0; b < CH / 8; ++b)
          tc_ld_32x32b_x8(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(h * HALF + c + 8 * b),
                          *reinterpret_cast<uint32_t(*)[8]>(v + 8 * b));
        tc_wait_ld();
#pragma unroll
        for (int e = 0; e < CH; ++e) {
          const int ml = h * HALF + c + e;  // row within the tile
          sts16(ystage + ml * 256 + row * 2, __half_as_ushort(__float2half_rn(__uint_as_float(v[e]))));
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
    if (P.silu) {
      // output jj of the rank's R columns pairs gate column 8(jj/4) + jj%4 with the one 4 later
      const int R2 = R >> 1;
      for (int it = threadIdx.x; it < R2 * BT; it += blockDim.x) {
        const int tok = it / R2, jj = it - tok * R2;
        const int rr = 8 * (jj >> 2) + (jj & 3);
        const int m = m0 + tok, n = n_base + rr;
        if (m >= P.M || n >= P.N) continue;
        float gt = 0.f, up = 0.f;
#pragma unroll 8
        for (int k = 0; k < S; ++k) {
          gt += red[(k * R + rr) * BT + tok];
          up += red[(k * R + rr + 4) * BT + tok];
        }
        P.Y[(size_t)m * (P.N >> 1) + (n_base >> 1) + jj] = __float2half_rn(silu_mul(gt, up));
      }
    }
    for (int it = threadIdx.x; it < (P.silu ? 0 : R * BT); it += blockDim.x) {
      const int tok = it / R, rr = it - tok * R;
      const int m = m0 + tok, n = n_base + rr;
      if (m >= P.M || n >= P.N) continue;
      float acc = 0.f;
#pragma unroll 8
      for (int k = 0; k < S; ++k) acc += red[(k * R + rr) * BT + tok];
      P.Y[(size_t)m * P.N + n] = __float2half_rn(acc);
    }
  }
  if (warp == 1 && lane == 0) {
    // No MMA may still run when TMEM is released.
    tc_wait_time_only(bar_acc, 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, SH::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------

cudaError_t tc_error_bits(uint32_t* bits, bool clear) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, s_err_tc, sizeof(v));
  if (e != cudaSuccess) return e;
  if (clear && v) {
    uint32_t zero = 0;
    e = cudaMemcpyToSymbol(s_err_tc, &zero, sizeof(zero));
  }
  *bits = v;
  return e;
}

namespace {

constexpr uint32_t kTcSmemMax = 227 * 1024;
constexpr int kTcMaxStages = 16;

// The kernel variants: (rows of X, units per ring slot, TMEM A slots).
struct TcVariant {
  int BT, KU, SB;
  uint32_t slot, tmem_cols;
};
template <int BT, int KU, int SB>
constexpr TcVariant tc_variant() {
  return {BT, KU, SB, TcShape<BT, KU, SB>::SLOT, TcShape<BT, KU, SB>::TMEM_COLS};
}
constexpr TcVariant kTcVariants[] = {
    tc_variant<16, 4, 3>(),  tc_variant<32, 4, 3>(),  tc_variant<64, 4, 3>(),  tc_variant<16, 2, 4>(),
    tc_variant<32, 2, 4>(),  tc_variant<64, 2, 4>(),  tc_variant<128, 2, 4>(), tc_variant<256, 2, 4>(),
};

// Units per ring slot: 4 (a super-group of g = 128) for small row tiles, where
// the per-slot hand-offs would otherwise dominate, 2 for the large ones.
bool tc_pick(int BT, int UPS, TcVariant* v) {
  const int KU = BT <= 64 ? std::min(4, UPS) : 2;
  for (const TcVariant& c : kTcVariants)
    if (c.BT == BT && c.KU == KU) {
      *v = c;
      return true;
    }
  return false;
}
uint32_t tc_bar_off(const TcVariant& v, int stages) { return v.slot * stages; }
uint32_t tc_smem_need(const TcVariant& v, int stages) {
  return tc_bar_off(v, stages) + 16 * (stages + v.SB) + 16 + 1024;
}

// Shared memory to request: at least what the ring needs, and enough that no
// more CTAs fit on an SM than tensor memory can hold at once (512 columns per
// SM), so that a tcgen05.alloc never waits on a CTA of the same cluster.
uint32_t tc_smem_request(int device, const TcVariant& v, int stages) {
  int per_sm = 0, reserved = 0;
  sm_shared_memory(device, &per_sm, &reserved);
  const int fit = 512 / (int)v.tmem_cols;  // CTAs whose TMEM fits on one SM
  const uint32_t floor_bytes = (uint32_t)(per_sm / (fit + 1) - reserved + 1024);
  return std::min<uint32_t>(kTcSmemMax, std::max(tc_smem_need(v, stages), floor_bytes));
}

template <int BT, int KU, int SB>
tm_status tc_launch_t(const CUtensorMap& tmX, const CUtensorMap& tmY, const tm_packed* p, const TcParams& P, int S,
                      uint32_t smem, cudaStream_t stream) {
  auto kern = tc_kernel<BT, KU, SB>;
  static std::atomic<unsigned long long> attr_done{0};  // one bit per device
  if (!smem_attr_once(attr_done, (const void*)kern, (int)kTcSmemMax)) return TM_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((P.NT + kTcTiles - 1) / kTcTiles), (unsigned)((P.M + BT - 1) / BT), (unsigned)S);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmX, p->tc_codes, p->tc_scales, p->tc_zeros, tmY, P);
  return e == cudaSuccess ? TM_OK : TM_ERR_CUDA;
}

int tc_tile_m_for(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256; }

}  // namespace

// Launch shape (fitted to GB300 measurements over the Llama-3 8B/70B
// shapes).  Every CTA holds all 512 tensor-memory columns, so one CTA runs per
// SM.  Rows of X per CTA: the smallest of 16/32/64/128/256 that holds M, halved
// (down to 64) while the output tiles would fill fewer than half the SMs --
// a tcgen05.mma costs about the same below N = 128, so narrow tiles buy
// parallelism cheaply.  K is split over a cluster (2 or 4 CTAs, never beyond
// one wave) only for row tiles up to 64, or for long K (>= 8192), where the
// reduction is cheap next to the K loop.  The ring is as deep as shared
// memory allows, up to 16 slots.
tm_status plan_tc(const tm_packed* p, int M, const tm_gemm_config* in, tm_gemm_config* out) {
  const Layout& L = p->L;
  if (in && in->tile_n && in->tile_n != 128) return TM_ERR_UNSUPPORTED;
  const int sms = num_sms(p->device);
  const int col_tiles = (L.NT + kTcTiles - 1) / kTcTiles;
  int BT = in && in->tile_m ? in->tile_m : tc_tile_m_for(M);
  if (!(in && in->tile_m))
    while (BT > 64 && col_tiles * ((M + BT - 1) / BT) < sms / 2) BT /= 2;
  TcVariant v;
  if (!tc_pick(BT, L.UPS, &v)) return TM_ERR_INVALID_ARG;
  const int want_S = in ? in->split_k : 0;
  if (want_S && want_S != 1 && want_S != 2 && want_S != 4 && want_S != 8) return TM_ERR_INVALID_ARG;
  const int rounds = L.Kp / kTcUnit / v.KU;  // ring slots of work over all of K
  int S = want_S;
  if (!S) {
    const int tiles = col_tiles * ((M + BT - 1) / BT);
    S = 1;
    if (BT <= 64 || L.K >= 8192)
      while (S < 4 && tiles * S * 2 <= sms && rounds / (S * 2) >= 2) S *= 2;
  }
  int stages = in && in->stages ? in->stages : 0;
  if (stages && (stages < 2 || stages > kTcMaxStages)) return TM_ERR_INVALID_ARG;
  if (!stages) {
    stages = kTcMaxStages;
    while (stages > 2 && tc_smem_need(v, stages) > kTcSmemMax) --stages;
  }
  if (tc_smem_need(v, stages) > kTcSmemMax) return TM_ERR_UNSUPPORTED;
  // the split-K receive buffer reuses the ring
  if (S > 1 && (uint32_t)kTcTiles * 16 * BT * 4 > v.slot * stages) return TM_ERR_UNSUPPORTED;
  out->path = 3;
  out->split_k = S;
  out->tile_n = 128;
  out->stages = stages;
  out->warp_n = 0;
  out->tile_m = BT;
  return TM_OK;
}

tm_status launch_tc(const void* X, const tm_packed* p, void* Y, int M, const tm_gemm_config& c,
                    cudaStream_t stream, bool silu) {
  const Layout& L = p->L;
  const int BT = c.tile_m;
  TcVariant v;
  if (!tc_pick(BT, L.UPS, &v)) return TM_ERR_UNSUPPORTED;
  CUtensorMap tmX;
  {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return TM_ERR_CUDA;
    cuuint64_t dims[2] = {(cuuint64_t)L.K, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)L.K * 2};
    cuuint32_t box[2] = {(cuuint32_t)kTcUnit, (cuuint32_t)BT};
    cuuint32_t es[2] = {1, 1};
    if (fn(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(X), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return TM_ERR_CUDA;
  }
  // the output as a tensor for the epilogue's TMA store: 128 columns x BT rows
  // (the fused silu form writes [M][N/2] with its own stores)
  CUtensorMap tmY;
  {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return TM_ERR_CUDA;
    const int ncols = silu ? L.N / 2 : L.N;
    cuuint64_t dims[2] = {(cuuint64_t)ncols, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)ncols * 2};
    cuuint32_t box[2] = {128u, (cuuint32_t)BT};
    cuuint32_t es[2] = {1, 1};
    if (fn(&tmY, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, Y, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return TM_ERR_CUDA;
  }
  TcParams P;
  P.Y = reinterpret_cast<__half*>(Y);
  P.M = M;
  P.N = L.N;
  P.NT = L.NT;
  P.UPS = L.UPS;
  P.g = L.g;
  P.kb_total = L.Kp / kTcUnit;
  const int S = c.split_k;
  const int rounds = P.kb_total / v.KU;
  P.kb_per_cta = ((rounds + S - 1) / S) * v.KU;
  P.stages = c.stages;
  P.bar_off = tc_bar_off(v, c.stages);
  P.silu = silu ? 1 : 0;
  if (tc_smem_need(v, c.stages) > kTcSmemMax) return TM_ERR_UNSUPPORTED;
  if ((uint32_t)BT * 256 > v.slot * (uint32_t)c.stages) return TM_ERR_UNSUPPORTED;  // the epilogue's staged tile
  const uint32_t smem = tc_smem_request(p->device, v, c.stages);
  tm_status st = TM_ERR_UNSUPPORTED;
  switch (BT * 16 + v.KU) {
    case 16 * 16 + 4: st = tc_launch_t<16, 4, 3>(tmX, tmY, p, P, S, smem, stream); break;
    case 32 * 16 + 4: st = tc_launch_t<32, 4, 3>(tmX, tmY, p, P, S, smem, stream); break;
    case 64 * 16 + 4: st = tc_launch_t<64, 4, 3>(tmX, tmY, p, P, S, smem, stream); break;
    case 16 * 16 + 2: st = tc_launch_t<16, 2, 4>(tmX, tmY, p, P, S, smem, stream); break;
    case 32 * 16 + 2: st = tc_launch_t<32, 2, 4>(tmX, tmY, p, P, S, smem, stream); break;
    case 64 * 16 + 2: st = tc_launch_t<64, 2, 4>(tmX, tmY, p, P, S, smem, stream); break;
    case 128 * 16 + 2: st = tc_launch_t<128, 2, 4>(tmX, tmY, p, P, S, smem, stream); break;
    case 256 * 16 + 2: st = tc_launch_t<256, 2, 4>(tmX, tmY, p, P, S, smem, stream); break;
    default: break;
  }
  if (st == TM_OK) set_launch_count(1);
  return st;
}

}  // namespace w4
