// Paged-latent MLA decode on CTA pairs (sm_103a), for bf16 rows loaded by TMA when a
// request's query rows come in groups of 128 (heads x draft tokens, e.g. 128 heads).
//
// The same computation as decode_sm103.cu — per query row, the softmax of
// sm_scale * <q, K_j> over the request's KV rows and its weighted sum of
// V_j = K_j[0:512] (the absorbed "data-movement friendly" MQA form of
// "mla_attention.py · tduncan/Nvidia-Optimization-Stack-VLLM", module docstring,
// over the paged cache of "Implementation:Sgl project Sglang Flash MLA", I/O
// Contract) — shaped for two SMs working as one tensor-core pair
// (tcgen05 .cta_group::2). A cluster of two CTAs takes a group of 128 query rows:
// CTA c holds query rows 64c .. 64c + 63 and, of every 128-row KV tile, rows
// 64c .. 64c + 63 (block 2t + c of the unit).
//   S = Q K^T   M = 128 (64 query rows per CTA) x N = 128 KV rows (64 from each
//               CTA's shared memory) x K = 576: 36 MMAs per tile. CTA c's accumulator
//               holds its 64 query rows against all 128 KV rows: TMEM lane r + 64h,
//               column n is row r against KV row n of tile half h.
//   O += P V    M = 128 (P of each CTA's 64 rows) x N = 256 value dims (each CTA
//               supplies 128 of them: dims 256b + 128c + 0..127) x K = 128 KV rows:
//               16 MMAs per tile for the 512 dims. CTA c's accumulator holds O of its
//               own 64 rows for all 512 dims: lane r + 64h, column 128b + d is dim
//               256b + 128h + d. Rescales and the epilogue therefore stay inside a CTA.
// Measured on GB300 with distinct operands and fully unrolled issue: the PV shape runs
// at the tensor cores' full rate per SM (64 cycles per K = 16 step), the S shape in 49
// cycles (about two thirds of it: the smallest pair instruction is bound by its issue);
// for the same query rows and KV rows the single-SM kernel needs twice the S instructions
// (M = 128 with 64 rows used, N = 64).
//
// Shared memory per CTA (224 KiB): Q (9 slabs of 64 rows x 64 dims, 128-B swizzle) and
// two stages of 9 dim slabs for the tile's KV rows, plus one 8-KiB P slab. A tile's stage
// first holds this CTA's 64 KV rows in all 576 dims: the S operand. The pair's B operand is
// split by N but its K dimension, the KV rows, is shared, so for PV each CTA needs V of all
// 128 rows for its own 256 value dims at offsets the two CTAs agree on: the slabs
// 4b + 2h + j hold tile half h's rows of the 64-dim slab j of this CTA's block-b dims.
// For the CTA's own half these are its S-operand slabs of its own value dims; the slabs of
// the peer's value dims are reloaded with the peer rows' values of this CTA's dims as soon
// as the S MMAs have read them. P of KV rows 0-63 goes to the RoPE slab, which S no longer
// needs; P of rows 64-127 to the extra slab. Tile t+1 loads into the other stage while tile
// t is computed.
//
// Warp roles (384 threads):
//   warp 0      TMA: Q once per unit and the S operand (completion counted on the even
//               CTA's barriers, which gate the MMAs); L2 prefetch of the next tile's rows
//   warp 1      TMEM allocation; TMA of the V operand (local barrier)
//   warp 2      S MMA issuer (even CTA only)
//   warp 3      PV MMA issuer (even CTA only)
//   warps 4-11  softmax (lane r + 64h: query row r over tile half h; warps 4-7 take S
//               columns 0-31 and O block 0, warps 8-11 columns 32-63 and O block 1),
//               O rescale, epilogue
#include <cstdint>
#include <cuda_runtime.h>

#include "decode_common.cuh"
#include "mla_kernels.h"
#include "ptx_sm103.cuh"

namespace mla {
namespace {

constexpr int kPairThreads = 384;
constexpr uint32_t kPSlab = 8192;  // 64 rows x 128 B
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffStage = kOffQ + 9 * kPSlab;       // 2 stages x 9 dim slabs of the tile's KV rows
constexpr uint32_t kStageBytes = 9 * kPSlab;
constexpr uint32_t kOffP1 = kOffStage + 2 * kStageBytes;  // P of KV rows 64-127 (rows 0-63: the stage's RoPE slab)
constexpr uint32_t kOffMisc = kOffP1 + kPSlab;
constexpr float kPairRescaleLog2 = 32.0f;
// A stage arrives in three parts of three dim slabs (slabs 3p .. 3p + 2), each on its own
// barrier, so that the S MMAs of the first slabs run while the later ones are still landing.
// S reads the slabs in order; the value slabs 4b + 2h + {0, 1} (block b, CTA h's dims) are
// released to the reload as a pair once slab 4b + 2h + 1 has been read.
constexpr int kStageParts = 3;

// Every barrier whose arrivals for tile t + 1 could come before its waiter has seen tile t
// is kept per stage (or per TMEM buffer): a parity wait must never be more than one phase
// behind.
enum PairBar {
  // gates of the MMA issuers, arrived on from both CTAs (used in the even CTA)
  kQFull = 0,       // count 2, + bytes
  kSRegFull = 1,    // + 3 * stage + part (2 x 3): count 2, + bytes
  kPFull = 7,       // count 16 (the softmax warps of both CTAs)
  kSFree = 8,       // + TMEM buffer (2): count 16
  kOFree = 10,      // count 16
  // signalled in both CTAs by the even CTA's multicast commits
  kSFull = 11,      // + TMEM buffer (2)
  kSDone = 13,      // + 4 * stage + 2 * b + h (2 x 4): S has read the slabs 4b + 2h + {0, 1}
  kStageFree = 21,  // + stage (2): the PV of the stage's tile has completed
  kPvDone = 23,
  kQEmpty = 24,
  kOFull = 25,
  // local to each CTA
  kVFull = 26,      // + stage (2): count 1, + bytes: this CTA's reload of the peer rows' values
  kFinal = 28,      // count 2: the last commit of each issuer (even CTA)
  kNumPairBars = 29
};

struct PairMisc {
  uint64_t bar[kNumPairBars];
  uint32_t tmem_base;
  int abort;
  int pad2;
  int pad;
  // the four threads of a query row exchange their tile maxima (slow path of a tile) and,
  // at the end of a unit, their partial sums here
  float xchg[256];
};
static_assert(kOffMisc + sizeof(PairMisc) + 1024 <= 232448, "shared memory budget of one CTA");

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    mla_decode_pair_kernel(const __grid_constant__ DecodeParams P, const __grid_constant__ CUtensorMap q_map,
                           const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ WideMaps wide) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_addr(smem);
  PairMisc* misc = reinterpret_cast<PairMisc*>(smem + kOffMisc);
  auto bar = [&](int i) -> uint32_t { return smem_addr(&misc->bar[i]); };
  volatile int* abort_flag = &misc->abort;
  auto stage = [&](int st) -> uint32_t { return sb + kOffStage + st * kStageBytes; };

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int c = static_cast<int>(rank);
  const bool leader = rank == 0;
  auto lead = [&](int i) -> uint32_t { return map_shared_rank(bar(i), 0); };  // the even CTA's barrier

  if (tid == 0) {
    mbar_init(bar(kQFull), 2);
    for (int s = 0; s < 2 * kStageParts; ++s) mbar_init(bar(kSRegFull + s), 2);
    mbar_init(bar(kPFull), 16);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kSFree + s), 16);
      mbar_init(bar(kSFull + s), 1);
      mbar_init(bar(kStageFree + s), 1);
      mbar_init(bar(kVFull + s), 1);
      for (int g = 0; g < 4; ++g) mbar_init(bar(kSDone + 4 * s + g), 1);
    }
    mbar_init(bar(kOFree), 16);
    mbar_init(bar(kPvDone), 1);
    mbar_init(bar(kQEmpty), 1);
    mbar_init(bar(kOFull), 1);
    mbar_init(bar(kFinal), 2);
    misc->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(&misc->tmem_base), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any remote arrive
  tc_fence_after();
  pdl_trigger();
  pdl_wait();
  const uint32_t tmem = misc->tmem_base;
  const uint32_t tmem_o = tmem;        // O: 2 blocks x 128 columns
  const uint32_t tmem_s = tmem + 256;  // S: 2 buffers x 64 columns

  const int R = P.rows_per_req;
  const int PG = R >> 7;  // groups of 128 query rows per request
  const int num_work = P.num_partitions * PG;
  const int cl0 = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(num_clusters_x());
  const int box_rows = P.page_size < kBlockRows ? P.page_size : kBlockRows;
  const int nbox = kBlockRows / box_rows;

  // pages of block `blk` of request r (-1: no rows to load); reports bad entries
  auto block_pages = [&](int r, int blk, int hi, int L, int* pages) -> int {
    int n = 0;
    for (int k = 0; k < nbox; ++k) {
      const int pos0 = blk * kBlockRows + k * box_rows;
      int page = -1;
      if (blk < hi && pos0 < L) {
        const int pi = pos0 >> P.log2_ps;
        page = pi < P.max_pages ? P.block_table[(int64_t)r * P.max_pages + pi] : -1;
        if (page < 0 || page >= P.num_pages) {
          atomicOr(P.status, 2u);
          page = -1;
        }
      }
      pages[k] = page;
      n += page >= 0;
    }
    return n;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ Q and S-operand loads
    // Tile t goes to stage t % 2 once the PV of tile t - 2 has released it; each slab group
    // completes on the even CTA's barrier for that group (both CTAs' bytes).
    if (lane == 0) {
      const bool wide_maps = wide.valid != 0;
      if (wide_maps) {
        tma_prefetch_desc(&wide.q9);
        tma_prefetch_desc(&wide.kv3);
      } else {
        tma_prefetch_desc(&q_map);
        tma_prefetch_desc(&kv_map);
      }
      int it = 0, u = 0;
      for (int w = cl0; w < num_work && !*abort_flag; w += ncl) {
        const int part = w / PG, g = w % PG;
        for_each_unit(P, part, [&](int r, int lo, int hi, int) {
          if (*abort_flag) return;
          if (u > 0 && !mbar_wait_cluster(bar(kQEmpty), (u - 1) & 1, abort_flag, P.status)) return;
          mbar_arrive_expect_tx_cluster(lead(kQFull), 9 * kPSlab);
          const int row0 = r * R + g * 128 + 64 * c;
          if (wide_maps) {
            tma_load_3d_pair(sb + kOffQ, &wide.q9, 0, row0, 0, lead(kQFull));  // all 9 slabs in one copy
          } else {
            for (int s = 0; s < 9; ++s) tma_load_2d_pair(sb + kOffQ + s * kPSlab, &q_map, s * 64, row0, lead(kQFull));
          }
          ++u;
          const int L = request_len(P, r);
          for (int b0 = lo; b0 < hi; b0 += 2, ++it) {
            const int st = it & 1;
            if (it >= 2 && !mbar_wait_cluster(bar(kStageFree + st), ((it >> 1) - 1) & 1, abort_flag, P.status)) return;
            int pages[8];
            const int own = b0 + c;
            const int nvalid = block_pages(r, own, hi, L, pages);
            for (int pt = 0; pt < kStageParts; ++pt)
              mbar_arrive_expect_tx_cluster(lead(kSRegFull + kStageParts * st + pt),
                                            static_cast<uint32_t>(3 * nvalid * box_rows * 128));
            if (wide_maps) {
              // page_size >= 64: the block is one page run, each part of 3 slabs one copy
              if (pages[0] >= 0)
                for (int pt = 0; pt < kStageParts; ++pt)
                  tma_load_4d_pair(stage(st) + 3 * pt * kPSlab, &wide.kv3, 0, (own * kBlockRows) & (P.page_size - 1),
                                   3 * pt, pages[0], lead(kSRegFull + kStageParts * st + pt));
            } else {
              for (int s = 0; s < 9; ++s)
                for (int k = 0; k < nbox; ++k) {
                  if (pages[k] < 0) continue;
                  const int in_page = (own * kBlockRows + k * box_rows) & (P.page_size - 1);
                  tma_load_3d_pair(stage(st) + s * kPSlab + k * box_rows * 128, &kv_map, s * 64, in_page, pages[k],
                                   lead(kSRegFull + kStageParts * st + s / 3));
                }
            }
            // Streams this CTA's rows of the unit's next tile from HBM into L2 (a hint; one bulk
            // prefetch per page box). Measured on the 128-head bf16 workload: one tile ahead
            // shortens the S-operand loads by a third; two tiles ahead gains nothing more, and
            // four or more slow the kernel (L2 thrashing).
            if (own + 2 < hi) {
              const int nxt = own + 2;
              for (int k = 0; k < nbox; ++k) {
                const int pos0 = nxt * kBlockRows + k * box_rows;
                if (pos0 >= L) break;
                const int pi = pos0 >> P.log2_ps;
                const int page = pi < P.max_pages ? P.block_table[static_cast<int64_t>(r) * P.max_pages + pi] : -1;
                if (page < 0 || page >= P.num_pages) continue;
                const int rows = (L - pos0) < box_rows ? (L - pos0) : box_rows;
                prefetch_l2_bulk(P.kv + static_cast<int64_t>(page) * P.page_bytes +
                                     static_cast<int64_t>(pos0 & (P.page_size - 1)) * P.row_bytes,
                                 static_cast<uint32_t>(rows * P.row_bytes));
              }
            }
          }
        });
      }
      if (*abort_flag && leader) {
        // copies still in flight land on this CTA's gates: wait for them (bounded)
        if (u > 0) mbar_wait_drain_cluster(bar(kQFull), (u - 1) & 1);
        for (int k = 1; k <= 2 && it - k >= 0; ++k)
          for (int pt = 0; pt < kStageParts; ++pt)
            mbar_wait_drain_cluster(bar(kSRegFull + kStageParts * ((it - k) & 1) + pt), ((it - k) >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ reload of the peer rows' values
    // The PV MMAs read V of both tile halves at the slabs 4b + 2h + j of the stage (h: the
    // half, b: the 256-dim block, j: the 64-dim slab of this CTA's 128 dims). For this CTA's
    // own half these are its own rows' S-operand slabs of its value dims; for the peer's half
    // they are the slabs of the peer's value dims, which S no longer needs once their group
    // of S MMAs has completed: they are reloaded with the peer rows' values of this CTA's dims.
    if (lane == 0) {
      int it = 0;
      for (int w = cl0; w < num_work && !*abort_flag; w += ncl) {
        const int part = w / PG;
        for_each_unit(P, part, [&](int r, int lo, int hi, int) {
          if (*abort_flag) return;
          const int L = request_len(P, r);
          for (int b0 = lo; b0 < hi; b0 += 2, ++it) {
            const int st = it & 1;
            const int h = 1 - c;  // the peer's half
            int pages[8];
            for (int b = 0; b < 2; ++b) {
              // the slabs 4b + 2h + {0, 1} are free once S has read them
              if (!mbar_wait_cluster(bar(kSDone + 4 * st + 2 * b + h), (it >> 1) & 1, abort_flag, P.status)) return;
              if (b == 0) {
                // (only now: S of this tile has begun, so the stage's previous reload has landed
                // and been waited for, and this arrival opens the barrier's next phase)
                const int n = block_pages(r, b0 + h, hi, L, pages);
                mbar_arrive_expect_tx(bar(kVFull + st), 4u * n * box_rows * 128);
              }
              if (wide.valid) {
                // one copy of 2 dim slabs: this CTA's dims of block b
                if (pages[0] >= 0)
                  tma_load_4d(stage(st) + (4 * b + 2 * h) * kPSlab, &wide.kv2, 0,
                              ((b0 + h) * kBlockRows) & (P.page_size - 1), 4 * b + 2 * c, pages[0], bar(kVFull + st));
              } else {
                for (int j = 0; j < 2; ++j) {
                  const int dst_slab = 4 * b + 2 * h + j;
                  const int src_slab = 4 * b + 2 * c + j;  // this CTA's value dims
                  for (int k = 0; k < nbox; ++k) {
                    if (pages[k] < 0) continue;
                    const int in_page = ((b0 + h) * kBlockRows + k * box_rows) & (P.page_size - 1);
                    tma_load_3d(stage(st) + dst_slab * kPSlab + k * box_rows * 128, &kv_map, src_slab * 64, in_page,
                                pages[k], bar(kVFull + st));
                  }
                }
              }
            }
          }
        });
      }
      if (*abort_flag)
        for (int k = 1; k <= 2 && it - k >= 0; ++k) mbar_wait_drain(bar(kVFull + ((it - k) & 1)), ((it - k) >> 1) & 1);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ S issuer (even CTA)
    if (leader && lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
      const uint64_t kmaj = sdesc_sw128(0, 16, 1024);
      const uint64_t qa = kmaj | ((sb + kOffQ) >> 4);
      int it = 0, u = 0;
      for (int w = cl0; w < num_work && !*abort_flag; w += ncl) {
        const int part = w / PG;
        for_each_unit(P, part, [&](int, int lo, int hi, int) {
          if (*abort_flag) return;
          if (!mbar_wait_cluster(bar(kQFull), u & 1, abort_flag, P.status)) return;
          for (int b0 = lo; b0 < hi; b0 += 2, ++it) {
            const int st = it & 1;
            if (it >= 2 && !mbar_wait_cluster(bar(kSFree + st), ((it >> 1) - 1) & 1, abort_flag, P.status)) return;
            tc_fence_after();
            const uint32_t d = tmem_s + st * 64;
            const uint64_t ka = kmaj | (stage(st) >> 4);
            // Fully unrolled, so that the descriptors are the base plus constants: an MMA issued
            // from a loop that computes its descriptors costs about 70 cycles, unrolled about 50.
#pragma unroll
            for (int pt = 0; pt < kStageParts; ++pt) {
              if (!mbar_wait_cluster(bar(kSRegFull + kStageParts * st + pt), (it >> 1) & 1, abort_flag, P.status))
                return;
              tc_fence_after();
#pragma unroll
              for (int i = 0; i < 3; ++i) {
                const int s = 3 * pt + i;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_bf16_pair(d, qa + s * (kPSlab >> 4) + kk * 2, ka + s * (kPSlab >> 4) + kk * 2, idesc_s,
                                (s | kk) ? 1u : 0u);
                // value slabs 4b + 2h + {0, 1} read: the reloader may overwrite them
                if (s < 8 && (s & 1)) mma_commit_pair(bar(kSDone + 4 * st + (s >> 1)), 3);
              }
            }
            // (failure-detection test: withhold the first tile's signal so that the
            // softmax's bounded wait runs out)
            if (!(P.test_withhold_signal && it == 0)) mma_commit_pair(bar(kSFull + st), 3);
          }
          mma_commit_pair(bar(kQEmpty), 3);
          ++u;
        });
      }
      mma_commit_pair(bar(kFinal), 1);
      mbar_wait_drain_cluster(bar(kFinal), 0);
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ PV issuer (even CTA)
    if (leader && lane == 0) {
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, 256, 0, 1);  // A = P (K-major), B = V (MN-major)
      const uint64_t kmaj = sdesc_sw128(0, 16, 1024);
      const uint64_t vmaj = sdesc_sw128(0, kPSlab, 1024);
      const uint64_t p1 = kmaj | ((sb + kOffP1) >> 4);
      int it = 0, u = 0;
      for (int w = cl0; w < num_work && !*abort_flag; w += ncl) {
        const int part = w / PG;
        for_each_unit(P, part, [&](int, int lo, int hi, int) {
          if (*abort_flag) return;
          for (int b0 = lo; b0 < hi; b0 += 2, ++it) {
            const int st = it & 1;
            const bool first = b0 == lo;
            if (!mbar_wait_cluster(bar(kPFull), it & 1, abort_flag, P.status)) return;
            if (first && u > 0 && !mbar_wait_cluster(bar(kOFree), (u - 1) & 1, abort_flag, P.status)) return;
            tc_fence_after();
            const uint64_t p0 = kmaj | ((stage(st) + 8 * kPSlab) >> 4);  // P of KV rows 0-63: the RoPE slab
            const uint64_t vb = vmaj | (stage(st) >> 4);
#pragma unroll
            for (int b = 0; b < 2; ++b) {
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const int h = k >> 2;
                const uint64_t a = (h ? p1 : p0) + (k & 3) * 2;
                const uint64_t bv = vb + (4 * b + 2 * h) * (kPSlab >> 4) + (k & 3) * (2048 >> 4);
                mma_bf16_pair(tmem_o + b * 128, a, bv, idesc_o, (first && k == 0) ? 0u : 1u);
              }
            }
            mma_commit_pair(bar(kPvDone), 3);
            mma_commit_pair(bar(kStageFree + st), 3);
          }
          mma_commit_pair(bar(kOFull), 3);
          ++u;
        });
      }
      mma_commit_pair(bar(kFinal), 1);
      mbar_wait_drain_cluster(bar(kFinal), 0);
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ softmax / epilogue
    // Lane wt = r + 64h of TMEM holds query row r (of this CTA's 64) against KV tile half
    // h in S, and dims 256b + 128h + 0..127 of that row in O. Two warps share each
    // 32-lane quarter (a warp reaches the lanes 32 (warp % 4) .. + 31): column group
    // cg = 0 takes S columns 0-31 and O block 0, cg = 1 columns 32-63 and O block 1. The
    // four threads of a row meet through shared memory; the eight warps meet at named
    // barrier 1 (no time limit: a thread whose bounded wait fails marks itself dead and
    // all stop together at the next barrier).
    const int sx = tid - 128;  // 0 .. 255
    const int cg = sx >> 7;
    const int wt = sx & 127;
    const int r = wt & 63;
    const int half = wt >> 6;
    const uint32_t lane_off = static_cast<uint32_t>(wt & ~31) << 16;
    bool dead = false, stop = false;
    auto wait = [&](uint32_t b, uint32_t parity) {
      if (!dead && !mbar_wait_cluster(b, parity, abort_flag, P.status)) dead = true;
      return !dead;
    };
    int it = 0, u = 0;
    for (int w = cl0; w < num_work && !stop; w += ncl) {
      const int part = w / PG, g = w % PG;
      const int grow = g * 128 + 64 * c + r;  // query row within the request
      const int tok = grow / P.heads;
      for_each_unit(P, part, [&](int rq, int lo, int hi, int sidx) {
        if (stop) return;
        const int L = request_len(P, rq);
        int lim = L;
        if (P.causal) {
          lim = L - P.sq + tok + 1;
          lim = lim > L ? L : lim;
        }
        const int end_unit = hi * kBlockRows;
        const int row_end = lim < end_unit ? lim : end_unit;  // KV positions < row_end count
        const int v_end = L < end_unit ? L : end_unit;        // rows < v_end hold loaded values
        float m_run = -INFINITY, l_run = 0.f;
        for (int b0 = lo; b0 < hi; b0 += 2, ++it) {
          const int st = it & 1;
          const bool first = b0 == lo;
          uint32_t sr[32];
          wait(bar(kSFull + st), (it >> 1) & 1);
          if (!dead) {
            tc_fence_after();
            tmem_ld32(tmem_s + st * 64 + lane_off + cg * 32, sr);
            tmem_wait_ld();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(lead(kSFree + st));
          const int pos0 = (b0 + half) * kBlockRows + cg * 32;  // KV position of this thread's column 0
          int nv = row_end - pos0;
          nv = nv < 0 ? 0 : (nv > 32 ? 32 : nv);
          const uint32_t vmask = nv == 32 ? ~0u : ((1u << nv) - 1u);
          float x[32];
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) {
            x[cc] = ((vmask >> cc) & 1u) ? __uint_as_float(sr[cc]) : -INFINITY;
            m4[cc & 3] = fmaxf(m4[cc & 3], x[cc]);
          }
          const float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * P.scale_log2;
          // the running maximum of a row moves (lazily) only when a tile exceeds it by more
          // than kPairRescaleLog2 powers of two; the four threads of the row take the same
          // decision
          const bool raise = mt > m_run + kPairRescaleLog2;
          float m_new = m_run;
          const bool any = named_bar_or(1, 256, raise || dead);
          if (any) {
            if (named_bar_or(1, 256, dead)) {
              stop = true;
              return;
            }
            misc->xchg[sx] = mt;
            named_bar_sync(1, 256);
            const float mh = fmaxf(fmaxf(misc->xchg[r], misc->xchg[r + 64]),
                                   fmaxf(misc->xchg[128 + r], misc->xchg[128 + r + 64]));
            m_new = (mh > m_run + kPairRescaleLog2) ? mh : m_run;
          }
          const bool rescale = any && !first && m_new != m_run && m_run != -INFINITY;
          const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
          const float alpha = fast_exp2(m_run - m_use);
          float ps4[4] = {0.f, 0.f, 0.f, 0.f};
          uint32_t pk[16];
#pragma unroll
          for (int cc = 0; cc < 16; ++cc) {
            const float p0 = fast_exp2(fmaf(x[2 * cc], P.scale_log2, -m_use));
            const float p1 = fast_exp2(fmaf(x[2 * cc + 1], P.scale_log2, -m_use));
            ps4[cc & 3] += p0 + p1;
            pk[cc] = f32x2_to_bf16x2(p0, p1);
          }
          l_run = l_run * alpha + ((ps4[0] + ps4[1]) + (ps4[2] + ps4[3]));
          m_run = m_new;
          // P of KV rows 64-127 and O belong to the previous tile's PV until it completes
          if (it > 0) wait(bar(kPvDone), (it - 1) & 1);
          if (any && !first && !dead) {
            // one TMEM round trip per 32 columns of this thread's 128 O columns
            tc_fence_after();
            const float a = rescale ? alpha : 1.0f;
#pragma unroll 1
            for (int k = 0; k < 4; ++k) {
              uint32_t t32[32];
              const uint32_t ta = tmem_o + lane_off + cg * 128 + k * 32;
              tmem_ld32(ta, t32);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) t32[i] = __float_as_uint(__uint_as_float(t32[i]) * a);
              tmem_st32(ta, t32);
            }
            tmem_wait_st();
            tc_fence_before();
          }
          if (!dead) {
            // P row r: KV rows of tile half `half`, 64 bf16 along K (K-major, 128-B swizzle),
            // of which this thread holds the 16-B chunks 4 cg .. 4 cg + 3; half 0 goes to the
            // stage's RoPE slab, which S has finished with
            const uint32_t pa = (half ? sb + kOffP1 : stage(st) + 8 * kPSlab) + r * 128;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              st_shared_v4(pa + (((4 * cg + q4) ^ (r & 7)) << 4),
                           make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]));
          }
          // the peer rows' values of this CTA's dims have landed; rows past the loaded range may
          // hold stale or non-finite bytes: zero them (their P is 0, and 0 x NaN would not be)
          wait(bar(kVFull + st), (it >> 1) & 1);
          if (!dead && (b0 + 2) * kBlockRows > v_end) {
            for (int hh = 0; hh < 2; ++hh) {
              int z0 = v_end - (b0 + hh) * kBlockRows;
              z0 = z0 < 0 ? 0 : z0;
              const int nz = (kBlockRows - z0) * 4 * 8;  // rows x slabs x 16-B chunks
              for (int idx = sx; idx < nz; idx += 256) {
                const int rr = z0 + idx / 32;
                const int j = (idx >> 3) & 3;
                const int ch = idx & 7;
                const int slab = 4 * (j >> 1) + 2 * hh + (j & 1);
                st_shared_v4(stage(st) + slab * kPSlab + rr * 128 + ch * 16, make_uint4(0, 0, 0, 0));
              }
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && !dead) mbar_arrive_cluster(lead(kPFull));
        }
        // -------------------------------------------------------- epilogue
        named_bar_sync(1, 256);  // every thread has read the last tile's maxima
        misc->xchg[sx] = l_run;
        if (named_bar_or(1, 256, dead)) {
          stop = true;
          return;
        }
        const float l_tot = (misc->xchg[r] + misc->xchg[r + 64]) + (misc->xchg[128 + r] + misc->xchg[128 + r + 64]);
        const int base_split = P.num_splits[rq];
        const int nsplit = P.num_splits[rq + 1] - base_split;
        const int sg = base_split + sidx;
        float inv = 0.f, lse2 = -INFINITY;
        if (l_tot > 0.f) {
          float denom = l_tot;
          if (nsplit == 1 && P.sink != nullptr) denom += fast_exp2(P.sink[grow % P.heads] * 1.4426950408889634f - m_run);
          inv = 1.0f / denom;
          lse2 = m_run + log2f(l_tot);
        }
        if (half == 0 && cg == 0) {
          const float lse_nat = lse2 * 0.6931471805599453f;
          if (nsplit == 1) P.lse[(int64_t)rq * R + grow] = lse_nat;
          else P.part_lse[(int64_t)sg * R + grow] = lse_nat;
        }
        if (wait(bar(kOFull), u & 1)) {
          tc_fence_after();
          // A warp holds 32 consecutive output rows (one per lane) and, per TMEM load, the same
          // 32 value dims of each. Eight rows at a time pass through this warp's 1-KiB slice of
          // the P slab (free here: the unit's last PV has completed; 16-B chunk q of staged row i
          // at position q ^ i), so that each global store covers contiguous dims of one row
          // (a store of one 16-B chunk per lane would touch 32 rows).
          const uint32_t xb = sb + kOffP1 + static_cast<uint32_t>(warp - 4) * 1024u;
          const int64_t row0 = (nsplit == 1 ? (int64_t)rq : (int64_t)sg) * R + (grow - lane);
#pragma unroll 1
          for (int k = 0; k < 4; ++k) {
            uint32_t t32[32];
            tmem_ld32(tmem_o + lane_off + cg * 128 + k * 32, t32);
            tmem_wait_ld();
            const int d0 = cg * 256 + half * 128 + k * 32;  // first value dim of these 32 columns
#pragma unroll
            for (int rnd = 0; rnd < 4; ++rnd) {
              if ((lane >> 3) == rnd) {
                const uint32_t i = static_cast<uint32_t>(lane & 7);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                  st_shared_v4(xb + i * 128 + ((static_cast<uint32_t>(q) ^ i) << 4),
                               make_uint4(__float_as_uint(__uint_as_float(t32[4 * q]) * inv),
                                          __float_as_uint(__uint_as_float(t32[4 * q + 1]) * inv),
                                          __float_as_uint(__uint_as_float(t32[4 * q + 2]) * inv),
                                          __float_as_uint(__uint_as_float(t32[4 * q + 3]) * inv)));
              }
              __syncwarp();
              if (nsplit == 1) {
                // bf16: 16 lanes per row, two dims each, two rows per store
                const int m = lane & 15;
#pragma unroll
                for (int i2 = 0; i2 < 8; i2 += 2) {
                  const uint32_t i = static_cast<uint32_t>(i2 + (lane >> 4));
                  const float2 v = ld_shared_v2f32(xb + i * 128 + ((static_cast<uint32_t>(m >> 1) ^ i) << 4) + (m & 1) * 8);
                  reinterpret_cast<uint32_t*>(P.out + (row0 + rnd * 8 + i) * 512 + d0)[m] = f32x2_to_bf16x2(v.x, v.y);
                }
              } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const float v = ld_shared_f32(xb + i * 128 + ((static_cast<uint32_t>(lane >> 2) ^ i) << 4) + (lane & 3) * 4);
                  P.part_out[(row0 + rnd * 8 + i) * 512 + d0 + lane] = v;
                }
              }
              __syncwarp();
            }
          }
          tc_fence_before();
        }
        __syncwarp();
        if (lane == 0 && !dead) mbar_arrive_cluster(lead(kOFree));
        ++u;
      });
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the even CTA's MMAs into both CTAs' TMEM have completed
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, 512);
}

}  // namespace

size_t decode_pair_smem_bytes() { return kOffMisc + sizeof(PairMisc) + 1024; }

cudaError_t launch_decode_pair(const DecodeParams& p, const CUtensorMap& q_map, const CUtensorMap& kv_map,
                               const WideMaps& wide, int clusters, cudaStream_t stream) {
  auto kern = mla_decode_pair_kernel;
  const size_t smem = decode_pair_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(2 * clusters), dim3(kPairThreads), smem, stream, p, q_map, kv_map, wide);
}

cudaError_t decode_pair_max_clusters(int* clusters) {
  auto kern = mla_decode_pair_kernel;
  const size_t smem = decode_pair_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms & ~1);
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(clusters, kern, &cfg);
}

}  // namespace mla
