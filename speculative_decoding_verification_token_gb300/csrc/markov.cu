// markov.cu -- DSpark Markov-head drafting (dspark_markov_draft).
//
// For every draft position k = 1..K (left to right, because row k depends on the token sampled at
// k - 1) two kernels run on the caller's stream:
//   position  persistent, warp-specialised CTAs, each owning a 128-request block and a strided
//             set of 64-column vocabulary tiles.  The CTA gathers the 128 rows U[x_{k-1}] (the
//             GEMM's A operand, 64 KB, kept in shared memory for every tile) and then pipelines:
//               warp 0      tensor-TMA loads of the Wt tile (64 vocabulary rows x 256) and of the
//                           backbone tile (128 requests x 64 columns) into a two-stage ring;
//               warp 1      tcgen05.mma (M = 128, N = 64, K = 256) into one of two TMEM
//                           accumulators;
//               warps 2-17  the epilogue, 16 columns of 32 requests per warp and tile: TMEM ->
//                           registers, + backbone, round to bf16 and staged in shared memory
//                           (three tiles deep), and
//                           per request: log2-domain softmax statistics and the exponential race
//                           x_k = argmax z - log(-log u) (DRAFT tag, position k) behind a noise
//                           gate whose bound is shared by every CTA of the row through a global
//                           table; one partial per (request, CTA).
//               warp 18     TMA stores of the staged z, one per lane quadrant (32 requests x
//                           64 columns) and tile.
//   select    folds the partials of every request into x_k, the row statistics of z_k and the
//             sequential-temperature-scaled confidence conf_k = 1 / (1 + exp(-s_k / T_k)).
#include <algorithm>
#include <cstring>
#include <mutex>

#include "race.cuh"
#include "sv_device.cuh"
#include "sv_host.h"
#include "tc.cuh"
#include "tmap.h"

namespace sv {

constexpr int kMkRows = 128;                 // requests per M-block (UMMA M)
constexpr int kMkCols = 64;                  // vocabulary columns per tile (UMMA N)
constexpr int kMkRank = 256;                 // R (UMMA K)
constexpr int kMkKB = kMkRank / 64;          // 128-byte k-blocks per row
constexpr int kMkStages = 2;                 // Wt / backbone ring depth
constexpr int kMkEpiWarps = 16;            // 4 lane quadrants x 4 column quarters
constexpr int kMkStoreWarp = 2 + kMkEpiWarps;       // issues the z stores
constexpr int kMkThreads = 32 * (3 + kMkEpiWarps);
constexpr int kMkZBufs = 3;                          // z staging depth (tiles)
constexpr uint32_t kMkABytes = kMkKB * kMkRows * 128;     // 64 KB
constexpr uint32_t kMkBBytes = kMkKB * kMkCols * 128;     // 32 KB per stage
constexpr uint32_t kMkBBBytes = kMkRows * 128;            // 16 KB per stage (64 bf16 per row)
constexpr uint32_t kMkZGroupBytes = 32 * 128;             // a lane quadrant's z block: 32 x 64 bf16
constexpr uint32_t kMkZBytes = kMkZBufs * 4 * kMkZGroupBytes;  // [buffer][quadrant]: 48 KB
constexpr size_t kMkSmem = 1024 + kMkABytes + kMkStages * (kMkBBytes + kMkBBBytes) + kMkZBytes;
constexpr uint32_t kMkTmemCols = 2 * kMkCols;             // two accumulators

struct MkPartial {  // one (request, CTA) partial of position k
  float m2;         // log2-domain running maximum
  float s;          // sum of 2^(z log2e - m2)
  float zmax;       // largest z
  float key;        // best race key
  int32_t idx;      // its vocabulary index
  int32_t pad[3];
};

struct MkParams {
  const void* U;              // bf16 [V][R]
  const int32_t* anchor;      // [B]
  int32_t* tokens;            // [B][K] drafted tokens (x_{k-1} read from here for k > 1)
  int32_t B, K, k;            // k: 1-based position
  int64_t V;
  int32_t n_mblocks, per_mblock, n_tiles;
  uint64_t seed;
  const uint64_t* request_ids;
  int32_t write_z;
  MkPartial* partials;        // [B][per_mblock]
  uint32_t* k0;               // [B] best exact race key published for row b so far (key_order; 0: none)
  int32_t* status;
};

__device__ __forceinline__ float bf16_round_f(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

struct KeyIdx {
  float key;
  int32_t idx;
};

// Exact race keys of the entries flagged in `surv` (bit j: column c0 + j of this thread's 16
// columns) against the running best; their z is read back from the staged block `tile` (two
// 16-byte chunks, cq and cq + 1, of the 128-byte swizzled row r).  Rare: out of line.
__device__ __noinline__ KeyIdx markov_survivors(Stream st, uint32_t surv, int64_t c0, int64_t V,
                                                const uint8_t* tile, uint32_t r, uint32_t cq,
                                                KeyIdx best) {
  while (surv) {
    const uint32_t j = __ffs(surv) - 1;
    surv &= surv - 1;
    const int64_t e = c0 + j;
    if (e >= V) continue;
    const uint16_t zbits =
        *reinterpret_cast<const uint16_t*>(tile + tc::sw128(r, cq + (j >> 3)) + 2 * (j & 7));
    const float z = __uint_as_float(uint32_t(zbits) << 16);
    if (!(z > -INFINITY)) continue;
    const uint4 blk = stream_block(st, static_cast<uint32_t>(e >> 3));
    const float u = race_uniform_at(st, static_cast<uint64_t>(e),
                                    half_of(blk, static_cast<uint32_t>(e & 7)));
    const float key = z + race_noise(u);
    if (race_better(key, static_cast<int32_t>(e), best.key, best.idx)) {
      best.key = key;
      best.idx = static_cast<int32_t>(e);
    }
  }
  return best;
}

// z = bf16(acc + backbone) for 16 columns: packed bf16 pairs for the store, fp32 values for the
// statistics and the race.  `valid` < 16 (the tile that crosses V) sets the columns from `valid`
// on to -inf: they hold zero-filled operands.
__device__ __forceinline__ void markov_round(float* v, const uint4& bb0, const uint4& bb1,
                                             int valid, uint32_t* zp) {
  const uint32_t bw[8] = {bb0.x, bb0.y, bb0.z, bb0.w, bb1.x, bb1.y, bb1.z, bb1.w};
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    const float2 zs = add2(make_float2(v[j], v[j + 1]), bf16x2_f2(bw[j / 2]));
    const __nv_bfloat162 z2 = __float22bfloat162_rn(zs);
    zp[j / 2] = *reinterpret_cast<const uint32_t*>(&z2);
    const float2 zf = bf16x2_f2(zp[j / 2]);
    v[j] = zf.x;
    v[j + 1] = zf.y;
  }
  if (valid < 16) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j >= valid) v[j] = -INFINITY;
  }
}

template <int kDummy = 0>
__global__ void __launch_bounds__(kMkThreads, 1)
    markov_position_kernel(const __grid_constant__ CUtensorMap map_wt,
                           const __grid_constant__ CUtensorMap map_bb,
                           const __grid_constant__ CUtensorMap map_z, MkParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + kMkABytes;                          // [stage][kb] 8 KB tiles
  uint8_t* sBB = sB + kMkStages * kMkBBytes;             // [stage] 16 KB
  uint8_t* sZ = sBB + kMkStages * kMkBBBytes;            // [buffer][quadrant] 4 KB
  __shared__ uint64_t b_full[kMkStages], b_empty[kMkStages];
  __shared__ uint64_t bb_full[kMkStages], bb_empty[kMkStages];
  __shared__ uint64_t acc_full[2], acc_empty[2];
  __shared__ uint64_t z_full[kMkZBufs], z_empty[kMkZBufs];
  __shared__ uint32_t tmem_base;
  __shared__ float merge[3][kMkRows][5];  // column quarters 1..3 -> quarter 0
  __shared__ int32_t s_bad;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t mb = blockIdx.x % p.n_mblocks;
  const int32_t ci = blockIdx.x / p.n_mblocks;
  const int32_t m0 = mb * kMkRows;
  const int32_t n_my = ci < p.n_tiles ? (p.n_tiles - ci + p.per_mblock - 1) / p.per_mblock : 0;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Wt and backbone tiles of tile t into ring stage t % kMkStages (producer thread only).  Wt is
  // read again at every position and by both M-blocks: keep it in L2 ahead of the backbone, which
  // is read once.
  auto issue_wt = [&](int t) {
    const int32_t n = ci + t * p.per_mblock;
    const int s = t % kMkStages;
    mbar_expect_tx(&b_full[s], kMkBBytes);
    for (int kb = 0; kb < kMkKB; ++kb)
      tc::tma_load_2d_hint(sB + s * kMkBBytes + kb * (kMkCols * 128), &map_wt, kb * 64,
                           n * kMkCols, &b_full[s], tc::policy_evict_last());
  };
  auto issue_bb = [&](int t) {
    const int32_t n = ci + t * p.per_mblock;
    const int s = t % kMkStages;
    mbar_expect_tx(&bb_full[s], kMkBBBytes);
    tc::tma_load_3d_hint(sBB + s * kMkBBBytes, &map_bb, n * kMkCols, p.k - 1, m0, &bb_full[s],
                         tc::policy_evict_first());
  };

  if (tid == 0) {
    s_bad = 0;
    for (int s = 0; s < kMkStages; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
      mbar_init(&bb_full[s], 1);
      mbar_init(&bb_empty[s], kMkEpiWarps);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kMkEpiWarps);
    }
    for (int z = 0; z < kMkZBufs; ++z) {
      mbar_init(&z_full[z], kMkEpiWarps);
      mbar_init(&z_empty[z], 1);
    }
    fence_barrier_init();
    // The first stages hold Wt and backbone tiles, which no kernel of this call writes: they are
    // requested before the wait for the previous position's tokens
    for (int t = 0; t < kMkStages && t < n_my; ++t) {
      issue_wt(t);
      issue_bb(t);
    }
  }
  if (warp == 1) tc::tmem_alloc(&tmem_base, kMkTmemCols);
  // A programmatic dependent of the previous position's select kernel: x_{k-1} and the partials
  // it reads are touched only after it has finished.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // A operand: the 128 rows U[x_{k-1}] in the swizzled K-major layout (rows past B use row 0)
  {
    const uint8_t* U = static_cast<const uint8_t*>(p.U);
    for (int c = tid; c < kMkRows * (kMkRank / 8); c += kMkThreads) {
      const int r = c / (kMkRank / 8);       // tile row
      const int ch = c % (kMkRank / 8);      // 16-byte chunk along K (0..31)
      const int32_t b = m0 + r;
      int32_t x = 0;
      if (b < p.B) {
        x = p.k == 1 ? p.anchor[b] : p.tokens[size_t(b) * p.K + (p.k - 2)];
        if (x < 0 || int64_t(x) >= p.V) {
          s_bad = 1;
          x = 0;
        }
      }
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(U + size_t(x) * (kMkRank * 2)) + ch);
      const int kb = ch >> 3;
      *reinterpret_cast<uint4*>(sA + kb * (kMkRows * 128) + tc::sw128(r, ch & 7)) = v;
    }
  }
  fence_proxy_async();  // the gathered rows are read by the tensor cores (async proxy)
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (tid == 0 && s_bad) report(p.status, SV_ERR_BAD_INPUT);
  const uint32_t tmem = tmem_base;

  if (warp == 0) {
    // ---- producer
    if (lane == 0) {
      for (int t = kMkStages; t < n_my; ++t) {  // tiles 0 .. kMkStages - 1 were issued above
        const int s = t % kMkStages;
        const uint32_t use = t / kMkStages;
        if (!mbar_wait(&b_empty[s], (use - 1) & 1, p.status)) break;
        issue_wt(t);
        if (!mbar_wait(&bb_empty[s], (use - 1) & 1, p.status)) break;
        issue_bb(t);
      }
    }
  } else if (warp == 1) {
    // ---- tensor-core issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kMkRows, kMkCols);
      const uint32_t a_base = smem_addr(sA);
      for (int t = 0; t < n_my; ++t) {
        const int s = t % kMkStages;
        const int acc = t & 1;
        if (t >= 2 && !mbar_wait(&acc_empty[acc], ((t >> 1) - 1) & 1, p.status)) break;
        if (!mbar_wait(&b_full[s], (t / kMkStages) & 1, p.status)) break;
        tc::fence_after_sync();
        const uint32_t b_base = smem_addr(sB + s * kMkBBytes);
        for (int kb = 0; kb < kMkKB; ++kb)
          for (int ks = 0; ks < 4; ++ks)  // 16 K-elements (32 bytes) per instruction
            tc::mma_bf16(tmem + acc * kMkCols,
                         tc::smem_desc_sw128(a_base + kb * (kMkRows * 128) + ks * 32),
                         tc::smem_desc_sw128(b_base + kb * (kMkCols * 128) + ks * 32), idesc,
                         (kb | ks) != 0);
        tc::mma_commit(&b_empty[s]);
        tc::mma_commit(&acc_full[acc]);
      }
    }
  } else if (warp == kMkStoreWarp) {
    // ---- z stores: once the sixteen epilogue warps have staged tile t in buffer t % kMkZBufs,
    // store its four 32 x 64 quadrant blocks; once the stores of tile t - 1 have read their
    // buffer, hand that buffer back to the epilogue
    if (lane == 0 && p.write_z) {
      const uint64_t once = tc::policy_evict_first();  // z is written once, read by the caller
      for (int t = 0; t < n_my; ++t) {
        const int32_t n = ci + t * p.per_mblock;
        const int zb = t % kMkZBufs;
        if (!mbar_wait(&z_full[zb], (t / kMkZBufs) & 1, p.status)) break;
        for (int q = 0; q < 4; ++q)
          if (m0 + 32 * q < p.B)  // a block wholly past B has nothing to store
            tc::tma_store_3d_hint(&map_z, sZ + (zb * 4 + q) * kMkZGroupBytes, n * kMkCols,
                                  p.k - 1, m0 + 32 * q, once);
        tc::bulk_commit();
        tc::bulk_wait_read<1>();
        if (t > 0) mbar_arrive(&z_empty[(t - 1) % kMkZBufs]);
      }
      tc::bulk_wait_all();
    }
  } else {
    // ---- epilogue: warp w reads TMEM lane quadrant q = w % 4 (rows 32q .. 32q + 31) and column
    // quarter h (16 columns) of each 64-column tile; thread (q, lane) owns request m0 + 32q + lane.
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const uint32_t r = 32 * q + lane;
    const int32_t b = m0 + static_cast<int32_t>(r);
    const uint64_t req = b < p.B ? (p.request_ids ? p.request_ids[b] : uint64_t(b)) : 0;
    const Stream st = make_stream(p.seed, req, static_cast<uint32_t>(p.k), kTagDraft);
    // Row-wide race bound: every CTA that holds a column range of row b publishes its best exact
    // key there, and every thread gates its entries against the largest key published so far
    // (read one tile late, off the critical path).  Any published key is the key of an entry of
    // the row, so it never exceeds the row's maximum and the gate stays conservative.
    uint32_t* const kslot = b < p.B ? p.k0 + b : nullptr;
    uint32_t kpub = 0;            // key_order of the published bound read at the previous tile
    float published = -INFINITY;  // the largest key this thread has published
    float m2 = kM2Empty, s = 0.f, zmax = -INFINITY;
    KeyIdx best = {-INFINITY, -1};
    bool failed = false;
    for (int t = 0; t < n_my; ++t) {
      const int32_t n = ci + t * p.per_mblock;
      const int sb = t % kMkStages;
      const int acc = t & 1;
      float v[16];
      // the two coarse Philox blocks of this tile's 16 columns need no accumulator: written ahead
      // of the wait, so the compiler may schedule them into it (1.276 -> 1.251 ms per call)
      const int64_t c0 = int64_t(n) * kMkCols + h * 16;
      const uint4 cblk0 = stream_block(st, static_cast<uint32_t>(c0 >> 3));
      const uint4 cblk1 = stream_block(st, static_cast<uint32_t>(c0 >> 3) + 1);
      if (!failed && !mbar_wait(&acc_full[acc], (t >> 1) & 1, p.status)) failed = true;
      __syncwarp();
      tc::fence_after_sync();
      tc::tmem_load16(tmem + (uint32_t(32 * q) << 16) + acc * kMkCols + h * 16, v);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      if (!failed && !mbar_wait(&bb_full[sb], (t / kMkStages) & 1, p.status)) failed = true;
      const uint8_t* bt = sBB + sb * kMkBBBytes;
      const uint4 bb0 = *reinterpret_cast<const uint4*>(bt + tc::sw128(r, 2 * h));
      const uint4 bb1 = *reinterpret_cast<const uint4*>(bt + tc::sw128(r, 2 * h + 1));
      __syncwarp();
      if (lane == 0) mbar_arrive(&bb_empty[sb]);
      const int valid = static_cast<int>(p.V - c0 < 16 ? (p.V - c0 > 0 ? p.V - c0 : 0) : 16);
      uint32_t zp[8];
      markov_round(v, bb0, bb1, valid, zp);
      // stage the quadrant's 32 x 64 block of z (the four warps of lane quadrant q, one 16-column
      // quarter each): the source of its TMA store and of the survivors' re-read.  The buffer was
      // last read by the stores of tile t - kMkZBufs.
      const int zb = t % kMkZBufs;
      uint8_t* zt = sZ + (zb * 4 + q) * kMkZGroupBytes;
      if (p.write_z && t >= kMkZBufs) {
        if (!failed && !mbar_wait(&z_empty[zb], (t / kMkZBufs - 1) & 1, p.status)) failed = true;
        __syncwarp();
      }
      *reinterpret_cast<uint4*>(zt + tc::sw128(lane, 2 * h)) = make_uint4(zp[0], zp[1], zp[2], zp[3]);
      *reinterpret_cast<uint4*>(zt + tc::sw128(lane, 2 * h + 1)) =
          make_uint4(zp[4], zp[5], zp[6], zp[7]);
      // softmax statistics (log2 domain): one rescale per tile, then e_j = 2^(z_j log2e - m2)
      float tmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < 16; ++j) tmax = fmaxf(tmax, v[j]);
      zmax = fmaxf(zmax, tmax);
      const float vm = tmax * kLog2e;
      if (vm > m2) {
        s *= fast_exp2(m2 - vm);
        m2 = vm;
      }
      float2 e[8];  // e[i] = (e_{2i}, e_{2i+1})
      {
        const float2 l2 = splat2(kLog2e), nm = splat2(-m2);
#pragma unroll
        for (int i = 0; i < 8; ++i) e[i] = exp2_2(fma2(make_float2(v[2 * i], v[2 * i + 1]), l2, nm));
        const float2 t = add2(add2(add2(e[0], e[4]), add2(e[2], e[6])),
                              add2(add2(e[1], e[5]), add2(e[3], e[7])));
        s += t.x + t.y;
      }
      // exponential race, key z_j + G_j with G_j = -log(-log u_j).  K is the larger of this
      // thread's best key and the row bound.  Entry j can reach K only if G_j >= K - z_j; since
      // G <= -log(1 - u) and 1 - u > m_j 2^-23 with m_j >= (0xFFFF - h_j) << 7 for the coarse half
      // h_j of u_j, that needs (0xFFFF - h_j) << 7 <= 2^((z_j - K) log2e + 23)
      // = e_j 2^(m2 + 23 - K log2e).  The 1e-3 margin covers the binary32 rounding of both
      // sides; the few entries that pass draw their low bits and are keyed exactly
      // (markov_survivors).  The 16 columns' coarse halves are two Philox blocks.
      {
        if (best.idx < 0 && tmax > -INFINITY) {
          // first finite tile: seed K with the exact key of the tile's largest z
          uint32_t top = 0;
#pragma unroll
          for (int j = 0; j < 16; ++j) top |= (v[j] == tmax ? 1u : 0u) << j;
          best = markov_survivors(st, top, c0, p.V, zt, lane, 2 * h, best);
        }
        const float kp = key_from_order(kpub);
        const float K = fmaxf(best.key, kp);
        const float C = fast_exp2(m2 + 23.0f - K * kLog2e) * 1.001f;
        // First per block of 8 entries: the largest coarse half against the largest e_j C
        // rejects almost every block.  Within a block that passes, rej collects, most
        // significant first, the sign of e_j C - ((0xFFFF - h_j) << 7): set = rejected (fma
        // rounds the exact difference once, so its sign is exact).
        uint32_t surv = 0;  // bit j: entry j may beat K
        const float2 C2 = splat2(C);
        const float ecap = fast_exp2(vm - m2) * 1.001f * C;  // >= e_j C for each of the 16
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const uint4 blk = g == 0 ? cblk0 : cblk1;
          if (gate_mh(half_max(blk)) > ecap) continue;  // none of the block's 8 entries passes
          const uint32_t w4[4] = {blk.x, blk.y, blk.z, blk.w};
          uint32_t rej = 0;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // entries 8g + 2k (low half) and 8g + 2k + 1 (high half): -((0xFFFF - h) << 7) as
            // binary32, from -(2^23 + that integer) plus 2^23
            const float2 nmf =
                add2(make_float2(__uint_as_float(((w4[k] & 0xFFFFu) << 7) ^ 0xCB7FFF80u),
                                 __uint_as_float(((w4[k] >> 9) & 0x7FFF80u) ^ 0xCB7FFF80u)),
                     splat2(8388608.0f));
            const float2 d = fma2(e[4 * g + k], C2, nmf);
            rej = __funnelshift_l(__float_as_uint(d.x), rej, 1);
            rej = __funnelshift_l(__float_as_uint(d.y), rej, 1);
          }
          surv |= (__brev(~rej) >> 24) << (8 * g);
        }
        if (surv) best = markov_survivors(st, surv, c0, p.V, zt, lane, 2 * h, best);
        if (kslot) {
          if (best.key > published && best.key > kp) {
            atomicMax(kslot, key_order(best.key));
            published = best.key;
          }
          kpub = __ldcg(kslot);  // consumed at the next tile
        }
      }
      if (p.write_z) {
        fence_proxy_async();  // the staged block is read by the async proxy (TMA store)
        __syncwarp();
        if (lane == 0) mbar_arrive(&z_full[zb]);
      }
    }
    // fold the four column quarters of every request and publish this CTA's partial
    if (h > 0) {
      merge[h - 1][r][0] = m2;
      merge[h - 1][r][1] = s;
      merge[h - 1][r][2] = zmax;
      merge[h - 1][r][3] = best.key;
      merge[h - 1][r][4] = __int_as_float(best.idx);
    }
    named_sync(1, 32 * kMkEpiWarps);
    if (h == 0 && b < p.B) {
#pragma unroll
      for (int hh = 0; hh < 3; ++hh) {
        ms2_merge(m2, s, merge[hh][r][0], merge[hh][r][1]);
        zmax = fmaxf(zmax, merge[hh][r][2]);
        const int32_t i2 = __float_as_int(merge[hh][r][4]);
        if (race_better(merge[hh][r][3], i2, best.key, best.idx)) {
          best.key = merge[hh][r][3];
          best.idx = i2;
        }
      }
      MkPartial out;
      out.m2 = m2;
      out.s = s;
      out.zmax = zmax;
      out.key = best.key;
      out.idx = best.idx;
      out.pad[0] = out.pad[1] = out.pad[2] = 0;
      p.partials[size_t(b) * p.per_mblock + ci] = out;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kMkTmemCols);
  }
}

// One warp per request: fold the CTA partials of position k into x_k, the statistics of z_k and
// the confidence.  A row without a finite maximum or with a NaN / +inf entry reports BAD_INPUT
// and drafts token 0 (so the next position still reads a valid row of U).
__global__ void __launch_bounds__(256)
    markov_select_kernel(const MkPartial* __restrict__ partials, int32_t per, int32_t B,
                         int32_t K, int32_t k, const float* __restrict__ conf_scores,
                         const float* __restrict__ sts_T, int32_t* tokens, float* row_stats,
                         float* conf_out, int32_t* status) {
  // a programmatic dependent of the position kernel: its partials are read after it has finished
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int32_t b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (b >= B) return;
  float m2 = kM2Empty, s = 0.f, zmax = -INFINITY, key = -INFINITY;
  int32_t idx = -1;
  for (int32_t i = lane; i < per; i += 32) {
    const MkPartial pt = partials[size_t(b) * per + i];
    ms2_merge(m2, s, pt.m2, pt.s);
    zmax = fmaxf(zmax, pt.zmax);
    if (race_better(pt.key, pt.idx, key, idx)) {
      key = pt.key;
      idx = pt.idx;
    }
  }
  warp_ms2(m2, s);
  zmax = warp_max(zmax);
  warp_race(key, idx);
  if (lane == 0) {
    const size_t o = size_t(b) * K + (k - 1);
    const bool bad = idx < 0 || !(s > 0.f) || isinf(s) || !(zmax < INFINITY);
    if (bad) report(status, SV_ERR_BAD_INPUT);
    tokens[o] = bad ? 0 : idx;
    if (row_stats) {
      row_stats[2 * o] = zmax;
      row_stats[2 * o + 1] = (m2 + log2f(s)) * kLn2;
    }
    if (conf_out) conf_out[o] = 1.f / (1.f + expf(-conf_scores[o] / sts_T[k - 1]));
  }
}

// ---- host side --------------------------------------------------------------------------------
namespace {

struct MkGeom {
  int32_t n_mblocks, per_mblock, n_tiles;
};

// 128-request blocks x vocabulary tiles; one CTA per SM, the SMs split evenly between the blocks.
bool markov_geom(int32_t B, int64_t V, MkGeom* g) {
  const int sms = device_sm_count();
  if (sms <= 0) return false;
  g->n_mblocks = (B + kMkRows - 1) / kMkRows;
  g->n_tiles = static_cast<int32_t>((V + kMkCols - 1) / kMkCols);
  g->per_mblock = std::max(1, std::min(sms / std::max(1, g->n_mblocks), g->n_tiles));
  return true;
}

// [B][per_mblock] partials, then the [K][B] published race bounds
size_t markov_partials_bytes(int32_t B, const MkGeom& g) {
  return (size_t(B) * g.per_mblock * sizeof(MkPartial) + 255) & ~size_t(255);
}

size_t markov_ws_bytes(int32_t B, int32_t K, const MkGeom& g) {
  return markov_partials_bytes(B, g) + ((size_t(K) * B * sizeof(uint32_t) + 255) & ~size_t(255));
}

}  // namespace
}  // namespace sv

extern "C" size_t dspark_markov_workspace_bytes(int32_t B, int32_t K, int64_t V, int32_t R) {
  (void)R;
  sv::MkGeom g;
  if (B <= 0 || K < 1 || V <= 0 || !sv::markov_geom(B, V, &g)) return 0;
  return sv::markov_ws_bytes(B, K, g);
}

extern "C" sv_status dspark_markov_draft(const void* backbone_logits, int64_t ldb, const void* U,
                                         const void* Wt, int64_t ldw,
                                         const int32_t* anchor_token, const float* conf_scores,
                                         const float* sts_T, int32_t B, int32_t K, int64_t V,
                                         int32_t R, uint64_t seed, const uint64_t* request_ids,
                                         int32_t* draft_tokens, void* draft_logits_out,
                                         int64_t ldz, float* row_stats, float* conf_out,
                                         int32_t* status, void* workspace,
                                         size_t workspace_bytes, void* stream) {
  using namespace sv;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (B < 0 || K < 1 || K > SV_MAX_DRAFT_LEN || V < 1 || R < 1) return SV_ERR_INVALID;
  if (R != kMkRank || V > (int64_t(1) << 31) - kMkCols) return SV_ERR_UNSUPPORTED;
  if (!backbone_logits || !U || !Wt || !anchor_token || !draft_tokens) return SV_ERR_INVALID;
  if (conf_out && (!conf_scores || !sts_T)) return SV_ERR_INVALID;
  if (ldb < V || ldw < R || (draft_logits_out && ldz < V)) return SV_ERR_INVALID;
  if (ldb % 8 || ldw % 8 || (draft_logits_out && ldz % 8)) return SV_ERR_UNSUPPORTED;
  if (!aligned16(backbone_logits) || !aligned16(U) || !aligned16(Wt) ||
      (draft_logits_out && !aligned16(draft_logits_out)))
    return SV_ERR_UNSUPPORTED;
  if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), cs) != cudaSuccess)
    return SV_ERR_CUDA;
  if (B == 0) return SV_OK;
  MkGeom g;
  if (!markov_geom(B, V, &g)) return SV_ERR_CUDA;
  if (!workspace || !aligned256(workspace) || workspace_bytes < markov_ws_bytes(B, K, g))
    return SV_ERR_INVALID;

  // tensor maps: Wt [V][R]; backbone and z [B][K][V] with row (b, k) at (b K + k) ld elements
  CUtensorMap map_wt, map_bb, map_z;
  {
    const uint64_t dims[2] = {uint64_t(R), uint64_t(V)};
    const uint64_t strides[1] = {uint64_t(ldw) * 2};
    const uint32_t box[2] = {64, kMkCols};
    if (!make_map(&map_wt, Wt, 2, dims, strides, box)) return SV_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {uint64_t(V), uint64_t(K), uint64_t(B)};
    const uint64_t strides[2] = {uint64_t(ldb) * 2, uint64_t(ldb) * 2 * K};
    const uint32_t box[3] = {kMkCols, 1, kMkRows};
    if (!make_map(&map_bb, backbone_logits, 3, dims, strides, box)) return SV_ERR_CUDA;
  }
  if (draft_logits_out) {
    const uint64_t dims[3] = {uint64_t(V), uint64_t(K), uint64_t(B)};
    const uint64_t strides[2] = {uint64_t(ldz) * 2, uint64_t(ldz) * 2 * K};
    const uint32_t box[3] = {kMkCols, 1, 32};  // one lane quadrant's block
    if (!make_map(&map_z, draft_logits_out, 3, dims, strides, box)) return SV_ERR_CUDA;
  } else {
    map_z = map_bb;  // never used: write_z = 0
  }
  if (cudaFuncSetAttribute(markov_position_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kMkSmem)) != cudaSuccess)
    return SV_ERR_CUDA;

  MkParams p;
  p.U = U;
  p.anchor = anchor_token;
  p.tokens = draft_tokens;
  p.B = B;
  p.K = K;
  p.V = V;
  p.n_mblocks = g.n_mblocks;
  p.per_mblock = g.per_mblock;
  p.n_tiles = g.n_tiles;
  p.seed = seed;
  p.request_ids = request_ids;
  p.write_z = draft_logits_out != nullptr;
  p.partials = static_cast<MkPartial*>(workspace);
  uint32_t* const bounds = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) +
                                                       markov_partials_bytes(B, g));
  p.status = status;
  const int grid = g.n_mblocks * g.per_mblock;
  const int sel_grid = (B + 7) / 8;
  if (cudaMemsetAsync(bounds, 0, size_t(K) * B * sizeof(uint32_t), cs) != cudaSuccess)
    return SV_ERR_CUDA;
  profile_mark(0, cs);
  // every launch after the first is a programmatic dependent of the one before (it starts while
  // that one finishes and waits for it with griddepcontrol.wait before touching its outputs)
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t pos_cfg = {};
  pos_cfg.gridDim = dim3(grid);
  pos_cfg.blockDim = dim3(kMkThreads);
  pos_cfg.dynamicSmemBytes = kMkSmem;
  pos_cfg.stream = cs;
  cudaLaunchConfig_t sel_cfg = pos_cfg;
  sel_cfg.gridDim = dim3(sel_grid);
  sel_cfg.blockDim = dim3(256);
  sel_cfg.dynamicSmemBytes = 0;
  sel_cfg.attrs = pdl;
  sel_cfg.numAttrs = 1;
  for (int32_t k = 1; k <= K; ++k) {
    p.k = k;
    p.k0 = bounds + size_t(k - 1) * B;
    pos_cfg.attrs = k > 1 ? pdl : nullptr;
    pos_cfg.numAttrs = k > 1 ? 1 : 0;
    if (cudaLaunchKernelEx(&pos_cfg, markov_position_kernel<0>, map_wt, map_bb, map_z, p) !=
        cudaSuccess)
      return SV_ERR_CUDA;
    if (k == 1) profile_mark(1, cs);
    if (cudaLaunchKernelEx(&sel_cfg, markov_select_kernel,
                           static_cast<const MkPartial*>(p.partials), g.per_mblock, B, K, k,
                           conf_scores, sts_T, draft_tokens, row_stats, conf_out, status) !=
        cudaSuccess)
      return SV_ERR_CUDA;
    if (k == 1) profile_mark(2, cs);
  }
  profile_mark(3, cs);
  return launch_status(cudaGetLastError());
}
