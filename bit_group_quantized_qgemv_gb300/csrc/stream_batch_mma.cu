// stream_batch_mma.cu -- small-batch GEMV on the tensor cores,
// Y[m] = W . X[m] (+ R[m]) for M = 3..8 activation rows, and M = 2 on short
// ops (INFERENCE_RESEARCH.md section 1: routing by M; the weights are loaded
// once and applied to every row of the batch).
//
// At M > 1 the product is a real (if thin) dense contraction: every decoded
// weight meets M activations, and on CUDA cores the M fp32 FMAs per weight
// bound the kernel (about 8 FMAs per weight at M = 8).  Here the codes are
// decoded exactly as in the M = 1 kernel -- masked into fp16 subnormals
// q * 2^-24 (one AND per two codes) -- and fed as the A operand of
// mma.sync.m16n8k16 (f16 x f16 -> f32), 16 weight rows x 16 k per MMA, with
// the batch's activations as the B operand (n = 8 columns: batch rows).
// Code lanes that the masks leave scaled by 16 (4-bit) or 4, 16, 64 (2-bit)
// meet activations pre-divided by the same power of two, so one accumulator
// takes every class.  Per 64-k quantisation group the fp32 fragment is
// scaled and the bias term added on the CUDA cores:
//   acc += scale * sum(q x) + bias * sum(x)           (units of 2^-24)
// the FMA-reordered dequantisation of the hada.io page (topic 27758),
// factored per group as in the M = 1 kernel.
//
// Ring, producer and epilogue warps follow the streaming kernel.  Warp 0
// (the producer) copies stages of 16 rows x KC k with TMA tensor copies:
// the codes in one 3-D copy that views each row as 128-byte columns and
// lands them 128-byte swizzled, [column][16 rows][128 B], so the fragment
// loads of 8 rows are free of bank conflicts; plus 16 rows of scales and of
// biases (see chunked_layout).  8 consumer warps each take KC/8 of a stage's
// k; warp 1 (the epilogue) sums the consumer warps' partials of a 16-row
// tile in a fixed order, adds the residual and stores fp16.  Each CTA owns a
// band of whole 16-row tiles.  The activations are staged in shared memory,
// already in B-fragment order, with their per-group sums, by the consumer
// warps themselves (each stages the groups it will read, the first chunk
// before any math and chunk c + 1 around stage c of the first tile); they
// bound the batch a pass can hold (2 * M_pad * K bytes).
#include <cuda.h>

#include <mutex>

#include "qgemv_stream.cuh"

namespace qgemv {
namespace {

constexpr int kMmaWarps = 8;                 // consumer warps
constexpr int kTileRows = 16;                // rows of one MMA tile (and one stage)
constexpr int kXsBudget = 132 * 1024;        // activation fragments + group sums
// K is split over a cluster of 4 when one CTA would stage more than 96 KB
// of activations (every CTA takes in all of them beside its weights: a
// quarter each is cheaper than the exchange of partials), else kept whole
// unless it does not fit.  Measured on GB300 (graph replays, 4096 rows,
// 4-bit; whole / split in 2 / split in 4): K = 8192, M = 4 10.8 / 10.7 /
// 11.8 us (68 KB: kept whole), M = 8 13.8 / 12.2 / 11.8; K = 14336, M = 4
// 14.9 / 14.2 / 13.8, M = 8 (does not fit whole) 16.0 / 15.1; K = 16384,
// M = 8 21.5 / 19.7; K = 4096, M = 8 6.3 whole against 7.9 split in 2.
constexpr int kSplitAbove = 96 * 1024;
constexpr int kRedBytes = 2 * kMmaWarps * 32 * 16;  // two tiles of warp partials
constexpr int kSmemPerBlock = 227 * 1024;    // sm_100-family opt-in shared memory per block
// Dynamic shared memory of a CTA in a cluster of cl: what the block may
// hold less a bound on the kernel's static part (barriers, 384 bytes, and
// for cl > 1 the cluster exchange slots, 512 bytes per slot and rank); the
// ring takes all that the staged activations leave.
constexpr int kXSlots = 4;  // cluster exchange slots: ranks run up to 4 tiles ahead of rank 0
constexpr int dyn_smem_max(int cl) {
  return kSmemPerBlock - 512 - (cl > 1 ? kXSlots * 512 * cl : 0);
}
// Threads of a CTA: producer warp, epilogue warp, the consumer warps.
constexpr int kBlockThreads = 64 + 32 * kMmaWarps;
constexpr int kAlignSlack = 1024;            // the ring starts on a 1024-byte boundary
// From M = 3 up the tensor cores are faster than the CUDA-core small-batch
// kernel on every shape (graph replays on GB300, o_proj 4096x4096 + down
// 4096x14336, 4-bit: M = 4 19.8 against 25.6 us; M = 8 21.9 against 45.8).
// At M = 2 the CUDA-core kernel's 2 FMAs per weight are cheap and it
// streams long ops better, while the tensor-core kernel's shorter start
// wins on short ones: M = 2 takes the tensor cores only for K <= 4096 and
// at most kMma2Bytes of weights per SM (4096x4096 5.21 against 5.72 us,
// 6144x4096 6.61 / 7.10, 1024x1024 2.29 / 3.98, 3072x1024 3.55 / 4.18; but
// 14336x4096 11.14 / 10.88, 4096x8192 10.61 / 8.29, 4096x14336 13.62 /
// 11.65).
constexpr int kMmaMinM = 2;
constexpr long long kMma2Bytes = 128 * 1024;

// Geometry of one launch (host-side plan, passed to the kernel).
struct MmaGeom {
  int kc;          // k per stage (divides K)
  int ccb, csb;    // code / scale bytes of one row and stage
  int cswz;        // swizzle mask of the scale and bias boxes (see swz; chunked: unused)
  int stage_bytes, ns, smem_bytes, grid, prefill, tiles;
  int cl;          // CTAs per cluster splitting K (1, 2, 4)
};

// Offset of logical byte `o` of a box written by a swizzled TMA copy: the
// 16-byte chunk index (bits 4..6) is XORed with bits 7..9, as many of them
// as the swizzle span allows (mask 0x70: 128 B, 0x30: 64 B, 0x10: 32 B).
__device__ __forceinline__ int swz(int o, int mask) { return o ^ ((o >> 3) & mask); }

// Codes of one word as four (4-bit) or eight (2-bit) fp16-subnormal pairs
// (see dot_word4 / dot_word2): (q0, q4), 16 (q1, q5), (q2, q6), 16 (q3, q7).
__device__ __forceinline__ void decode_word4(uint32_t w, uint32_t (&v)[4]) {
  v[0] = w & 0x000F000Fu;
  v[1] = w & 0x00F000F0u;
  const uint32_t w8 = w >> 8;
  v[2] = w8 & 0x000F000Fu;
  v[3] = w8 & 0x00F000F0u;
}
__device__ __forceinline__ void decode_word2(uint32_t w, uint32_t (&v)[8]) {
  v[0] = w & 0x00030003u;
  v[1] = w & 0x000C000Cu;
  v[2] = w & 0x00300030u;
  v[3] = w & 0x00C000C0u;
  const uint32_t w8 = w >> 8;
  v[4] = w8 & 0x00030003u;
  v[5] = w8 & 0x000C000Cu;
  v[6] = w8 & 0x00300030u;
  v[7] = w8 & 0x00C000C0u;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// A 3-D box {x, y, z} of a tensor map into this CTA's shared memory,
// completion counted on `bar`.
__device__ __forceinline__ void tma_box3(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

// A 2-D box (x: byte column, y: row), likewise.
__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap* map, int x, int y,
                                        uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// ------------------------------------------------------------ clusters
// Rank of this CTA in its cluster, a shared-memory address of this CTA
// mapped to the same offset in rank `r`'s shared memory, a 16-byte store
// there, and a release arrive on an mbarrier there (cluster scope).
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t r) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(saddr), "r"(r));
  return out;
}
// 16 bytes into another CTA's shared memory, completing 16 bytes of the
// transaction count of that CTA's mbarrier (no fence, no arrive).
__device__ __forceinline__ void st_async_f4(uint32_t addr, float4 v, uint32_t remote_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::
          "r"(addr),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(remote_bar)
      : "memory");
}
__device__ __forceinline__ void arrive_remote(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}
// Bounded wait with cluster-scope acquire (for phases completed by other
// CTAs of the cluster); gives up after about one second like mbar_wait.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, unsigned* status) {
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, "
        "%3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(20000u)
        : "memory");
    if (ok) return true;
    if (global_timer_ns() - t0 > 1000000000ull) {
      atomicOr(status, kStatusWaitTimeout);
      return false;
    }
  }
}

// fp16 pair (low half of a, low half of b) or (high of a, high of b).
__device__ __forceinline__ uint32_t pair_lo(uint32_t a, uint32_t b) {
  return __byte_perm(a, b, 0x5410);
}
__device__ __forceinline__ uint32_t pair_hi(uint32_t a, uint32_t b) {
  return __byte_perm(a, b, 0x7632);
}

// Both halves times 2^-s (s = 0, 2, 4, 6), one fp16 rounding (exact unless
// the result is subnormal).
__device__ __forceinline__ uint32_t scale_pair(uint32_t v, int s) {
  if (s == 0) return v;
  const __half2 f = __float2half2_rn(s == 2 ? 0.25f : (s == 4 ? 0.0625f : 0.015625f));
  __half2 h = *reinterpret_cast<const __half2*>(&v);
  h = __hmul2(h, f);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// B-fragment registers of one lane (batch row m, t = lane % 4) for one
// 64-k group, from the 16 activations x[16t .. 16t+15] of that group held as
// 8 fp16 pairs w[j] = (x[2j], x[2j+1]).  MMA mi gets registers 2 mi, 2 mi+1.
//  4-bit: words 2t, 2t+1 of a row (k 16t .. 16t+15); MMA mi takes word
//         2t + mi/2, code lanes (q0,q4),(q2,q6) (mi even) or 16 (q1,q5),
//         16 (q3,q7) (mi odd, activations / 16).
//  2-bit: word t (k 16t .. 16t+15); MMA mi takes code class 4^mi: lanes
//         (c_mi, c_mi+8), (c_mi+4, c_mi+12), activations / 4^mi.
template <int BITS>
__device__ __forceinline__ void bfrag_group(const uint32_t (&w)[8], uint32_t (&b)[8]) {
  if (BITS == 4) {
#pragma unroll
    for (int mi = 0; mi < 4; ++mi)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int k0 = 8 * (mi >> 1) + (mi & 1) + 2 * r;  // pair (k0, k0 + 4)
        const uint32_t p = (k0 & 1) ? pair_hi(w[k0 >> 1], w[(k0 >> 1) + 2])
                                    : pair_lo(w[k0 >> 1], w[(k0 >> 1) + 2]);
        b[2 * mi + r] = scale_pair(p, (mi & 1) ? 4 : 0);
      }
  } else {
#pragma unroll
    for (int mi = 0; mi < 4; ++mi)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int k0 = mi + 4 * r;  // pair (k0, k0 + 8)
        const uint32_t p = (k0 & 1) ? pair_hi(w[k0 >> 1], w[(k0 >> 1) + 4])
                                    : pair_lo(w[k0 >> 1], w[(k0 >> 1) + 4]);
        b[2 * mi + r] = scale_pair(p, 2 * mi);
      }
  }
}

template <int BITS, int MP, bool CHUNKED, int CL>
__global__ void __launch_bounds__(kBlockThreads, 1)
    batch_mma_kernel(const StreamArgs a, const MmaGeom gm,
                     const __grid_constant__ CUtensorMap tm_codes,
                     const __grid_constant__ CUtensorMap tm_scales,
                     const __grid_constant__ CUtensorMap tm_biases) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t redfull_bar[2];
  __shared__ __align__(8) uint64_t redempty_bar[2];
  __shared__ __align__(8) uint64_t xready_bar;
  // cluster split of K (CL > 1): rank 0 collects the other ranks' tile
  // partials (cfull: rank 0's own arrive with the expected bytes, the other
  // ranks' asynchronous stores completing them) and hands the slots back
  // (cempty, on the other ranks)
  __shared__ __align__(8) uint64_t cfull_bar[kXSlots];
  __shared__ __align__(8) uint64_t cempty_bar[kXSlots];
  __shared__ __align__(16) float4 xred[CL > 1 ? kXSlots * CL * 32 : 1];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int K = a.K;
  const int M = a.M;
  const int N = static_cast<int>(a.rows);
  // Cluster split of K: rank r of a cluster of CL CTAs takes k in
  // [r K/CL, (r+1) K/CL) of the cluster's rows; the CTA's own k range is
  // what it stages, streams and reduces.
  const int rank = CL > 1 ? static_cast<int>(cluster_rank()) : 0;
  const int Kc = K / CL;
  const int kbase = rank * Kc;
  const int G = Kc / 64;                 // groups of this CTA's k range
  const int KC = gm.kc;
  const int NC = Kc / KC;                // chunks per row and CTA
  const int GPC = KC / 64;               // groups per chunk
  const int GPW = GPC / kMmaWarps;       // groups per consumer warp and stage
  const int NS = gm.ns;
  // this cluster's band of whole tiles
  const int ncl = static_cast<int>(gridDim.x) / CL;
  const int cid = static_cast<int>(blockIdx.x) / CL;
  const int t0 = static_cast<int>(static_cast<long long>(cid) * gm.tiles / ncl);
  const int t1 = static_cast<int>(static_cast<long long>(cid + 1) * gm.tiles / ncl);
  const int ntiles = t1 - t0;
  const int nstages = ntiles * NC;
  // Stage layout: the codes as [ccb / 128][16 rows][128 B], 128-byte
  // swizzled (2 KB per column, 1024-byte aligned), then the scales and the
  // biases: whole rows as swizzled boxes at 2 KB steps, chunks as plain
  // [16][csb] blocks (128-byte aligned).
  const int scales_off = kTileRows * gm.ccb;
  const int biases_off = scales_off + (CHUNKED ? ((kTileRows * gm.csb + 127) & ~127) : 2048);

  // shared memory: the ring (1024-byte aligned for the swizzled boxes), then
  // B fragments [G][2][4 MP][4 u32], group sums [G][8] fp32 (x 2^-24), and
  // two tiles of warp partials [2][W][32][4].
  uint8_t* ring = smem_raw + ((kAlignSlack - (smem_u32(smem_raw) & (kAlignSlack - 1))) &
                              (kAlignSlack - 1));
  uint4* xs_frag = reinterpret_cast<uint4*>(ring + static_cast<size_t>(NS) * gm.stage_bytes);
  float* xs_sum = reinterpret_cast<float*>(xs_frag + static_cast<size_t>(G) * 2 * 4 * MP);
  float4* red = reinterpret_cast<float4*>(xs_sum + static_cast<size_t>(G) * 8);

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), kMmaWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&redfull_bar[b]), kMmaWarps);
      mbar_init(smem_u32(&redempty_bar[b]), 1);
    }
    mbar_init(smem_u32(&xready_bar), kMmaWarps);
    for (int b = 0; b < kXSlots; ++b) {
      mbar_init(smem_u32(&cfull_bar[b]), 1);
      mbar_init(smem_u32(&cempty_bar[b]), 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (CL > 1) {
    // every CTA's barriers exist before any remote arrive (the CTAs of a
    // cluster run together, and none returns before this point)
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
  }

  // ------------------------------------------------------------ producer
  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      const uint32_t stage_tx =
          static_cast<uint32_t>(kTileRows) * static_cast<uint32_t>(gm.ccb + 2 * gm.csb);
      int slot = 0, issued = 0;
      uint32_t phase = 0;
      for (int st = 0; st < nstages; ++st) {
        const int tile = st / NC, c = st - tile * NC;
        const int row0 = (t0 + tile) * kTileRows;
        if (st == gm.prefill && !mbar_wait(smem_u32(&xready_bar), 0, &g_status)) break;
        if (!mbar_wait(smem_u32(&empty_bar[slot]), phase ^ 1u, &g_status)) break;
        const uint32_t fb = smem_u32(&full_bar[slot]);
        const uint32_t sb = smem_u32(ring + static_cast<size_t>(slot) * gm.stage_bytes);
        mbar_arrive_expect_tx(fb, stage_tx);  // rows past N arrive zero-filled, counted
        const int kb = kbase + c * KC;  // first k of the stage
        // all of the stage's codes in one copy: 128-byte columns j of 16 rows
        tma_box3(sb, &tm_codes, 0, row0, kb * BITS / 8 / 128, fb, pol);
        tma_box(sb + scales_off, &tm_scales, kb / 32, row0, fb, pol);
        tma_box(sb + biases_off, &tm_biases, kb / 32, row0, fb, pol);
        ++issued;
        if (++slot == NS) {
          slot = 0;
          phase ^= 1u;
        }
      }
      // Drain: never leave while a copy into this CTA's shared memory is in flight.
      for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j)
        mbar_wait(smem_u32(&full_bar[j % NS]), (j / NS) & 1, &g_status);
    }
    return;
  }

  const int g = lane >> 2, t = lane & 3;

  // Final values of a tile (lane: rows g, g + 8; batch rows 2t, 2t + 1),
  // scaled back from 2^-24, plus the residual, rounded to fp16 into y.
  auto store_tile = [&](int tile, const float (&v)[4]) {
    const int row0 = (t0 + tile) * kTileRows;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = row0 + g + ((i & 2) ? 8 : 0);
      const int m = 2 * t + (i & 1);
      if (row < N && m < M) {
        const size_t o = static_cast<size_t>(m) * N + row;
        float y = v[i] * kTwo24;
        if (a.residual != nullptr) y += __half2float(a.residual[o]);
        a.y[o] = __float2half_rn(y);
      }
    }
  };

  // ------------------------------------------------------------ epilogue
  if (warp == 1) {
    pdl_wait();  // residuals and y belong to the stream order
    for (int tile = 0; tile < ntiles; ++tile) {
      const int b = tile & 1;
      if (!mbar_wait(smem_u32(&redfull_bar[b]), (tile >> 1) & 1, &g_status)) return;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      for (int w = 0; w < kMmaWarps; ++w) {
        const float4 p = red[(b * kMmaWarps + w) * 32 + lane];
        v[0] += p.x;
        v[1] += p.y;
        v[2] += p.z;
        v[3] += p.w;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&redempty_bar[b]));
      if (CL > 1) {
        const int x = tile % kXSlots;                         // exchange slot
        const uint32_t xph = static_cast<uint32_t>(tile / kXSlots) & 1u;  // its phase
        if (rank != 0) {
          // hand this CTA's partial of the tile to rank 0 (slot x, once rank
          // 0 has read the tile kXSlots back from it)
          if (tile >= kXSlots &&
              !mbar_wait_cluster(smem_u32(&cempty_bar[x]), xph ^ 1u, &g_status))
            return;
          st_async_f4(map_to_rank(smem_u32(&xred[(x * CL + rank) * 32 + lane]), 0),
                      make_float4(v[0], v[1], v[2], v[3]), map_to_rank(smem_u32(&cfull_bar[x]), 0));
          continue;
        }
        // rank 0: add the other ranks' partials, in rank order, once their
        // (CL - 1) x 512 bytes have landed (the transaction count may run
        // ahead of this expectation; the phase needs both)
        if (lane == 0) mbar_arrive_expect_tx(smem_u32(&cfull_bar[x]), (CL - 1) * 32 * 16);
        if (!mbar_wait_cluster(smem_u32(&cfull_bar[x]), xph, &g_status)) return;
        for (int r = 1; r < CL; ++r) {
          const float4 p = xred[(x * CL + r) * 32 + lane];
          v[0] += p.x;
          v[1] += p.y;
          v[2] += p.z;
          v[3] += p.w;
        }
        __syncwarp();
        if (lane == 0 && tile + kXSlots < ntiles)  // the slot is reused: hand it back
          for (int r = 1; r < CL; ++r) arrive_remote(map_to_rank(smem_u32(&cempty_bar[x]), r));
      }
      store_tile(tile, v);
    }
    return;
  }

  // ----------------------------------------------------------- consumers
  const int cw = warp - 2;  // consumer warp 0..7
  pdl_wait();               // x may come from the previous kernel
  // Stage the activations, warp by warp: in every chunk of a stage a
  // consumer warp reads only the B fragments and group sums of its own
  // GPW groups (gi = c GPC + cw GPW + j), so it stages exactly those and no
  // warp waits for another.  A quad of lanes (t = 0..3) takes one (batch
  // row m, group): each lane reads its 16 activations (two 16-byte loads),
  // forms its 8 B-fragment registers and its part of the group sum; the quad
  // adds the four parts.  Rows m in [M, MP) are zero.  The first chunk is
  // staged before any stage is computed; chunk c + 1's loads are issued
  // before stage (tile 0, c) is computed and converted after it, so their
  // latency hides behind the math.  Every lane runs the same rounds, so the
  // quad shuffles always have all 32 lanes.
  constexpr int kRounds = MP;               // rounds per warp and chunk (GPW <= 8)
  const int items_w = MP * GPW * 4;
  const int rounds_w = (items_w + 31) / 32;
  uint4 raw[kRounds][2];
  auto stage_load = [&](int c) {
#pragma unroll
    for (int rd = 0; rd < kRounds; ++rd) {
      raw[rd][0] = raw[rd][1] = make_uint4(0u, 0u, 0u, 0u);
      const int i = rd * 32 + lane;  // i % 4 == t
      const int mg = i >> 2;
      const int m = mg / GPW, gi = c * GPC + cw * GPW + (mg - m * GPW);
      if (rd < rounds_w && i < items_w && m < M) {
        const uint4* src =
            reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(m) * K + kbase + gi * 64 + 16 * t);
        raw[rd][0] = src[0];
        raw[rd][1] = src[1];
      }
    }
  };
  auto stage_store = [&](int c) {
#pragma unroll
    for (int rd = 0; rd < kRounds; ++rd) {
      if (rd >= rounds_w) break;  // uniform across the warp
      const int i = rd * 32 + lane;
      const int mg = i >> 2;
      const int m = mg / GPW, gi = c * GPC + cw * GPW + (mg - m * GPW);
      const uint32_t w[8] = {raw[rd][0].x, raw[rd][0].y, raw[rd][0].z, raw[rd][0].w,
                             raw[rd][1].x, raw[rd][1].y, raw[rd][1].z, raw[rd][1].w};
      float part = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
        part += f.x + f.y;
      }
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
      uint32_t b[8];
      bfrag_group<BITS>(w, b);
      if (i < items_w) {
        uint4* dst = xs_frag + (static_cast<size_t>(gi) * 2) * (4 * MP) + m * 4 + t;
        dst[0] = make_uint4(b[0], b[1], b[2], b[3]);
        dst[4 * MP] = make_uint4(b[4], b[5], b[6], b[7]);
        if (t == 0) xs_sum[gi * 8 + m] = part * kTwoM24;
      }
    }
    if constexpr (MP < 8) {
      constexpr int kPad = 8 - MP;
      for (int z = lane; z < kPad * GPW; z += 32)  // group sums of the padding rows
        xs_sum[(c * GPC + cw * GPW + z / kPad) * 8 + MP + z % kPad] = 0.f;
    }
    __syncwarp();  // the warp's lanes read each other's fragments
  };
  stage_load(0);
  stage_store(0);
  if (lane == 0) mbar_arrive(smem_u32(&xready_bar));  // the producer's prefill gate

  const bool bl = lane < 4 * MP;  // lanes whose batch row g holds activations
  const int cmask = gm.cswz;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  int slot = 0;
  uint32_t phase = 0;
  for (int st = 0; st < nstages; ++st) {
    const int tile = st / NC, c = st - tile * NC;
    const bool next_x = (tile == 0 && c + 1 < NC);  // stage the next chunk around this one
    if (next_x) stage_load(c + 1);
    if (!mbar_wait(smem_u32(&full_bar[slot]), phase, &g_status)) return;
    const uint8_t* sb = ring + static_cast<size_t>(slot) * gm.stage_bytes;
    // Four groups in flight per warp hide more of the decode -> MMA -> scale
    // chain (graph replays on GB300: M = 4 o_proj + down 20.3 against 21.0
    // us); with K split over a cluster two did better (M = 8 down 16.1
    // against 16.4 us).
#pragma unroll(CL == 1 ? 4 : 2)
    for (int j = 0; j < GPW; ++j) {
      const int gl = cw * GPW + j;     // group within the chunk
      const int gi = c * GPC + gl;     // group within the row
      uint32_t A0[8], A8[8];           // decoded pairs of rows g and g + 8
      if (BITS == 4) {
        const uint8_t* box = sb + (gl >> 2) * 2048;
        const int col = (gl & 3) * 32 + t * 8;
        const uint8_t* p0 = box + swz(g * 128 + col, 0x70);
        const uint8_t* p8 = box + swz((g + 8) * 128 + col, 0x70);
        const uint2 w0 = *reinterpret_cast<const uint2*>(p0);
        const uint2 w8 = *reinterpret_cast<const uint2*>(p8);
        uint32_t v[4];
        decode_word4(w0.x, v);
        A0[0] = v[0];
        A0[1] = v[2];
        A0[2] = v[1];
        A0[3] = v[3];
        decode_word4(w0.y, v);
        A0[4] = v[0];
        A0[5] = v[2];
        A0[6] = v[1];
        A0[7] = v[3];
        decode_word4(w8.x, v);
        A8[0] = v[0];
        A8[1] = v[2];
        A8[2] = v[1];
        A8[3] = v[3];
        decode_word4(w8.y, v);
        A8[4] = v[0];
        A8[5] = v[2];
        A8[6] = v[1];
        A8[7] = v[3];
      } else {
        const uint8_t* box = sb + (gl >> 3) * 2048;
        const int col = (gl & 7) * 16 + t * 4;
        const uint8_t* p0 = box + swz(g * 128 + col, 0x70);
        const uint8_t* p8 = box + swz((g + 8) * 128 + col, 0x70);
        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(p0);
        const uint32_t w8 = *reinterpret_cast<const uint32_t*>(p8);
        uint32_t v[8];
        decode_word2(w0, v);
#pragma unroll
        for (int mi = 0; mi < 4; ++mi) {
          A0[2 * mi] = v[mi];
          A0[2 * mi + 1] = v[mi + 4];
        }
        decode_word2(w8, v);
#pragma unroll
        for (int mi = 0; mi < 4; ++mi) {
          A8[2 * mi] = v[mi];
          A8[2 * mi + 1] = v[mi + 4];
        }
      }
      uint4 bq0 = make_uint4(0u, 0u, 0u, 0u), bq1 = bq0;
      if (bl) {
        bq0 = xs_frag[(static_cast<size_t>(gi) * 2 + 0) * (4 * MP) + lane];
        bq1 = xs_frag[(static_cast<size_t>(gi) * 2 + 1) * (4 * MP) + lane];
      }
      const uint32_t B[8] = {bq0.x, bq0.y, bq0.z, bq0.w, bq1.x, bq1.y, bq1.z, bq1.w};
      float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int mi = 0; mi < 4; ++mi)
        mma16816(d, A0[2 * mi], A8[2 * mi], A0[2 * mi + 1], A8[2 * mi + 1], B[2 * mi],
                 B[2 * mi + 1]);
      const int s0 = CHUNKED ? g * gm.csb + 2 * gl : swz(g * gm.csb + 2 * gl, cmask);
      const int s8 = CHUNKED ? (g + 8) * gm.csb + 2 * gl : swz((g + 8) * gm.csb + 2 * gl, cmask);
      const float sg = __half2float(*reinterpret_cast<const __half*>(sb + scales_off + s0));
      const float sg8 = __half2float(*reinterpret_cast<const __half*>(sb + scales_off + s8));
      const float bg = __half2float(*reinterpret_cast<const __half*>(sb + biases_off + s0));
      const float bg8 = __half2float(*reinterpret_cast<const __half*>(sb + biases_off + s8));
      const float2 xs = *reinterpret_cast<const float2*>(xs_sum + gi * 8 + 2 * t);
      acc[0] = fmaf(sg, d[0], fmaf(bg, xs.x, acc[0]));
      acc[1] = fmaf(sg, d[1], fmaf(bg, xs.y, acc[1]));
      acc[2] = fmaf(sg8, d[2], fmaf(bg8, xs.x, acc[2]));
      acc[3] = fmaf(sg8, d[3], fmaf(bg8, xs.y, acc[3]));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[slot]));
    if (++slot == NS) {
      slot = 0;
      phase ^= 1u;
    }
    if (next_x) stage_store(c + 1);
    if (c == NC - 1) {  // the tile is complete: hand its partials to the epilogue
      const int b = tile & 1;
      if (!mbar_wait(smem_u32(&redempty_bar[b]), ((tile >> 1) & 1) ^ 1u, &g_status)) return;
      red[(b * kMmaWarps + cw) * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&redfull_bar[b]));
      acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    }
  }
}

// Stage layout of a shape.  Rows whose scales fit one 128-byte swizzled box
// row (K <= 4096, codes at most 2 KB) stream whole: a stage is 16 complete
// rows, scales and biases as swizzled boxes.  Longer rows (and any row
// split across a cluster) are cut into chunks of KC k, the longest multiple
// of 512 up to 4096 that divides the CTA's k range and leaves a ring of two
// stages; their scales and biases come as plain [16][KC/32] rows.  Either
// way the codes of a stage are one copy: the copy engine streams a few large
// copies much faster than many small ones (measured on GB300: one 1-D copy
// per ring slot reaches ~10 / 19 / 38 / 44 GB/s per SM at 4 / 8 / 16 /
// 32 KB; down 4096 x 14336 at M = 4: 16.7 us as 2 KB boxes, 14.8 us as one
// copy per stage).
// (K: the k range of one CTA.)
bool chunked_layout(int bits, int K, int cl) {
  return cl > 1 || K * bits / 8 > 2048 || K / 32 > 128;
}

// Bytes of one ring stage for rows of K k cut into chunks of kc.
int stage_bytes_for(int bits, int K, int kc, int cl) {
  const int ccb = kc * bits / 8, csb = kc / 32;
  if (chunked_layout(bits, K, cl))  // 1024-byte steps keep every stage's swizzle phase
    return (kTileRows * ccb + 2 * ((kTileRows * csb + 127) & ~127) + 1023) & ~1023;
  return kTileRows * ccb + 4096;
}

// Chunk length and ring depth for a CTA's k range of K (whole rows in one
// stage when they fit a swizzled stage).  Long rows take the longest chunk
// (a multiple of 512 up to 4096 that divides K) whose ring still holds two
// stages next to the staged activations: few large copies beat a deeper ring
// of small ones (measured on GB300, down 4096 x 14336 at M = 4: 32 KB stages
// two deep 15.3 us, 18 KB stages five deep 17.9 us; M = 8: 9 KB stages ten
// deep 24.3 against 16.1 us).  false when no chunk fits.
bool pick_chunk(int bits, int K, int cl, int xs_bytes, int* kc_out, int* stage_out, int* ns_out) {
  const int budget = dyn_smem_max(cl) - kAlignSlack - xs_bytes - kRedBytes;
  auto ring = [&](int kc) {
    const int n = budget / stage_bytes_for(bits, K, kc, cl);
    return n > kMaxStages ? kMaxStages : n;
  };
  int kc = 0;
  if (!chunked_layout(bits, K, cl)) {
    if (K % 512 == 0 && K >= 512 && ring(K) >= 2) kc = K;
  } else {
    for (int c = 4096; c >= 512 && kc == 0; c -= 512)  // at most 8 groups per warp and stage
      if (K % c == 0 && ring(c) >= 2) kc = c;
  }
  if (kc == 0) return false;
  *kc_out = kc;
  *stage_out = stage_bytes_for(bits, K, kc, cl);
  *ns_out = ring(kc);
  return true;
}

// The driver's cuTensorMapEncodeTiled, reached through the runtime.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// (looked up once, thread-safely; null when the driver does not provide it)
EncodeTiledFn encode_fn() {
  static const EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(f);
    cudaGetLastError();
    return static_cast<EncodeTiledFn>(nullptr);
  }();
  return fn;
}

// 2-D byte-tensor map of `rows` rows of `row_bytes` bytes, boxes of
// box_bytes x 16 rows with the given swizzle.
bool encode_rows(CUtensorMap* m, const void* base, long long rows, int row_bytes, int box_bytes,
                 CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dim[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
  const cuuint64_t stride[1] = {static_cast<cuuint64_t>(row_bytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_bytes),
                             static_cast<cuuint32_t>(kTileRows)};
  const cuuint32_t estride[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dim, stride, box,
            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D byte-tensor map of a code matrix seen as 128-byte columns: x the byte
// within a column (128), y the row (stride row_bytes), z the column (stride
// 128 B).  A box of {128, 16, ccb / 128} lands in shared memory as
// [column][row][128 B] with the 128-byte swizzle: the layout of 16-row x
// 128 B boxes laid side by side, delivered by one copy.
bool encode_code_columns(CUtensorMap* m, const void* base, long long rows, int row_bytes,
                         int ccb) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || row_bytes % 128 != 0 || ccb % 128 != 0 || ccb / 128 > 256) return false;
  const cuuint64_t dim[3] = {128, static_cast<cuuint64_t>(rows),
                             static_cast<cuuint64_t>(row_bytes / 128)};
  const cuuint64_t stride[2] = {static_cast<cuuint64_t>(row_bytes), 128};
  const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(kTileRows),
                             static_cast<cuuint32_t>(ccb / 128)};
  const cuuint32_t estride[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dim, stride, box,
            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Clusters of `cl` CTAs of kernel k that can be resident at once with smem
// bytes of dynamic shared memory (cudaOccupancyMaxActiveClusters), cached per
// (kernel, cluster size, shared memory, device); a failed query is not
// cached and reads as 0.
template <typename F>
int resident_clusters(F* k, int cl, int smem, int device) {
  struct Entry {
    const void* k;
    int cl, smem, device, n;
  };
  static std::mutex mu;
  static Entry cache[16] = {};
  static int next = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& e : cache)
    if (e.k == reinterpret_cast<const void*>(k) && e.cl == cl && e.smem == smem &&
        e.device == device)
      return e.n;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cl));
  cfg.blockDim = dim3(kBlockThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cl);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    return 0;
  }
  cache[next] = Entry{reinterpret_cast<const void*>(k), cl, smem, device, n};
  next = (next + 1) % 16;
  return n;
}

template <int BITS, int MP, bool CHUNKED, int CL>
cudaError_t launch_mma_t(const StreamArgs& a, MmaGeom gm, const CUtensorMap* maps,
                         cudaStream_t stream, int device) {
  static unsigned done_mask = 0;
  auto* k = batch_mma_kernel<BITS, MP, CHUNKED, CL>;
  cudaError_t e = ensure_smem_attr(k, dyn_smem_max(CL), &done_mask, device);
  if (e != cudaSuccess) return e;
  int clusters = gm.grid;  // one CTA per SM and cluster rank
  if (CL > 1) {
    const int n = resident_clusters(k, CL, gm.smem_bytes, device);
    if (n < 1) return cudaErrorNotSupported;
    clusters = gm.tiles < n ? gm.tiles : n;
  }
  gm.grid = clusters * CL;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(gm.grid));
  cfg.blockDim = dim3(kBlockThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(gm.smem_bytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(CL);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = CL > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k, a, gm, maps[0], maps[1], maps[2]);
}

}  // namespace

// Plan of the tensor-core small-batch kernel for M activation rows held in
// one pass (M_pad = 4 or 8 columns of the MMA's B operand); false when
// the shape does not fit (K not a multiple of 512, or the staged
// activations above their budget).
bool batch_mma_plan(int bits, int K, long long N, int M, int sms, int* mp_out, int* smem_out,
                    int* ns_out, int* cl_out, int* kc_out) {
  if ((bits != 4 && bits != 2) || M < kMmaMinM || M > kMaxM || N < 1 || sms < 1) return false;
  if (M == 2 && (K > 4096 || N * (static_cast<long long>(K) * bits / 8 + K / 32) > kMma2Bytes * sms))
    return false;
  const int mp = M <= 4 ? 4 : 8;
  // Split K across a cluster: into 4 when the activations of a whole row
  // are large (kSplitAbove), else only while one CTA cannot hold them.
  auto xs_of = [&](int c) { return 2 * mp * (K / c) + (K / c) / 2; };  // fragments + group sums
  auto splits = [&](int c) { return K % (c * 64 * kMmaWarps) == 0; };
  int cl = 1;
  if (xs_of(1) > kSplitAbove) cl = splits(4) ? 4 : (splits(2) ? 2 : 1);
  while (cl < 4 && xs_of(cl) > kXsBudget && splits(2 * cl)) cl *= 2;
  const int Kc = K / cl;
  if (Kc % (64 * kMmaWarps) != 0 || Kc < 64 * kMmaWarps) return false;
  const int xs_bytes = xs_of(cl);
  if (xs_bytes > kXsBudget) return false;
  int kc = 0, stage = 0, ns = 0;
  if (!pick_chunk(bits, Kc, cl, xs_bytes, &kc, &stage, &ns)) return false;
  *mp_out = mp;
  *smem_out = kAlignSlack + ns * stage + xs_bytes + kRedBytes;
  *ns_out = ns;
  *cl_out = cl;
  if (kc_out != nullptr) *kc_out = kc;
  return true;
}

cudaError_t stream_batch_mma(int bits, const StreamArgs& a, int sms, cudaStream_t st,
                             int device) {
  int mp = 0, smem = 0, ns = 0, cl = 1;
  if (!batch_mma_plan(bits, a.K, a.rows, a.M, sms, &mp, &smem, &ns, &cl))
    return cudaErrorNotSupported;
  MmaGeom gm{};
  gm.cl = cl;
  const int Kc = a.K / cl;
  const int xs_bytes = 2 * mp * Kc + Kc / 2;
  int stage = 0, ns2 = 0;
  if (!pick_chunk(bits, Kc, cl, xs_bytes, &gm.kc, &stage, &ns2) || ns2 != ns)
    return cudaErrorNotSupported;
  gm.ccb = gm.kc * bits / 8;
  gm.csb = gm.kc / 32;
  // scale / bias boxes: a swizzle span equal to the row when the row is 32,
  // 64 or 128 bytes, else none
  gm.cswz = gm.csb == 128 ? 0x70 : (gm.csb == 64 ? 0x30 : (gm.csb == 32 ? 0x10 : 0));
  gm.stage_bytes = stage;
  gm.ns = ns;
  gm.smem_bytes = smem;
  const long long tiles = (a.rows + kTileRows - 1) / kTileRows;
  gm.tiles = static_cast<int>(tiles);
  gm.grid = static_cast<int>(tiles < sms ? tiles : sms);
  gm.prefill = prefill_stages(gm.stage_bytes, ns);
  const bool chunked = chunked_layout(bits, Kc, cl);
  if (chunked) gm.cswz = 0;
  const CUtensorMapSwizzle ssw = gm.cswz == 0x70   ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : gm.cswz == 0x30 ? CU_TENSOR_MAP_SWIZZLE_64B
                                 : gm.cswz == 0x10 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                   : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUtensorMap maps[3];
  const int rcb = a.K * bits / 8, rgb = a.K / 32;
  const bool ok_maps =
      encode_code_columns(&maps[0], a.codes[0], a.rows, rcb, gm.ccb) &&
      encode_rows(&maps[1], a.scales[0], a.rows, rgb, gm.csb, ssw) &&
      encode_rows(&maps[2], a.biases[0], a.rows, rgb, gm.csb, ssw);
  if (!ok_maps) return cudaErrorInvalidValue;
#define QGEMV_MMA_LAUNCH(B, P)                                                  \
  return !chunked   ? launch_mma_t<B, P, false, 1>(a, gm, maps, st, device)  \
         : cl == 1  ? launch_mma_t<B, P, true, 1>(a, gm, maps, st, device)   \
         : cl == 2  ? launch_mma_t<B, P, true, 2>(a, gm, maps, st, device)   \
                    : launch_mma_t<B, P, true, 4>(a, gm, maps, st, device)
  if (bits == 4) {
    if (mp == 4) QGEMV_MMA_LAUNCH(4, 4);
    QGEMV_MMA_LAUNCH(4, 8);
  }
  if (mp == 4) QGEMV_MMA_LAUNCH(2, 4);
  QGEMV_MMA_LAUNCH(2, 8);
#undef QGEMV_MMA_LAUNCH
}

}  // namespace qgemv
