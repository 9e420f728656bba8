// Paged-latent MLA decode kernel for sm_103a (GB300).
//
// Computes, for every query row (token t, head n) of a request, the softmax of
// sm_scale * <q, K_j> over the request's candidate KV rows and its weighted sum
// of V_j = K_j[0:512] — the absorbed ("data-movement friendly", MQA) form of
// MLA ("mla_attention.py · tduncan/Nvidia-Optimization-Stack-VLLM", module
// docstring, "Data-Movement Friendly Approach") over a paged cache addressed
// through block_table ("Implementation:Sgl project Sglang Flash MLA", I/O
// Contract), with an optional per-head sink in the denominator ("MLA" API page
// of HALOps, mla_attention, attn_sink), causal draft tokens and top-k indices.
//
// One persistent CTA per SM processes work items (partition p, query group g):
// 64 query rows of one request against the KV blocks of the partition's
// segments. Per 64-row KV tile:
//   S   = Q K^T      tcgen05 MMA, M = 64 query rows (16 in each TMEM lane quarter),
//                    N = 64 KV rows, K = 576 / 512, fp32 accumulator in TMEM
//   P   = online softmax of S (exp2 domain, lazy rescale when the running max
//                    grows by more than kRescaleLog2), written as bf16 to shared memory
//   O^T += V^T P^T   tcgen05 MMA, M = 128 value dims (4 blocks), N = query rows,
//                    K = 64 KV rows, fp32 accumulator in TMEM (256 columns)
// The transposed output accumulator keeps O for 64 query rows x 512 dims in
// half of TMEM, leaving room for two S buffers so that S(j+1) overlaps the
// softmax of tile j.
//
// Warp roles (512 threads):
//   warp 0      TMA producer: Q once per unit, KV tiles through block_table (bf16 dense)
//   warp 1      TMEM allocator; L2 prefetch of upcoming tiles [layout 2 and bf16 gather: PV issuer]
//   warp 2      S MMA issuer (one thread)
//   warp 3      PV MMA issuer (one thread) [layout 2 and bf16 gather: L2 prefetch]
//   warps 4-7   softmax (16 query rows per warp, two threads per row) + O rescale + epilogue
//   warps 8-15  converters: fp8 -> bf16 dequantisation and sparse row gathers
#include <cstdint>
#include <cuda_runtime.h>

#include "decode_common.cuh"
#include "mla_kernels.h"
#include "ptx_sm103.cuh"

namespace mla {
namespace {

constexpr uint32_t kSlab = 8192;  // 64 rows x 128 B (64 bf16), SW128
constexpr int kNumBars = 40;
enum Bar {
  kQFull = 0,
  kQEmpty = 1,
  kKvFull = 2,    // + stage * 9 + group: slabs 4g..4g+3 (TMA path); [stage][0] for the converter path
  kKvEmpty = 20,  // + stage * 5 + k: V slabs 2k, 2k+1 free (k < 4); k = 4: the whole stage free
  kSFull = 30,    // +buffer
  kSFree = 32,    // +buffer
  kPFull = 34,    // +stage
  kPvDone = 36,
  kOFull = 37,
  kOFree = 38,
  kFinal = 39
};
__device__ __forceinline__ int kv_full(int st, int grp) { return kKvFull + st * 9 + grp; }
// TMA path: the S issuer checks one barrier per group of 4 slabs (each check stalls it
// until its queued MMAs are dispatched, so fewer checks keep the tensor pipe busier).
__device__ __forceinline__ int slab_group(int s) { return s >> 2; }
__device__ __forceinline__ int kv_empty(int st, int k) { return kKvEmpty + st * 5 + k; }
// Bytes of KV data the prefetch warp keeps in flight ahead of the stage fills.
constexpr uint32_t kPrefetchBytes = 160u * 1024u;  // 96-224 KB measured alike; 640 KB 4 % slower (DSV3)
// Lazy rescale: P = 2^(s - m) is taken against the running maximum m, which is
// raised (and O^T rescaled in TMEM) only when a tile's maximum exceeds it by
// more than this many powers of two. P then stays below 2^64 (bf16 and fp32 reach
// 2^128), the running sum below rows x 2^64, and O^T below rows x 2^64 x max|V|,
// inside fp32 while rows x max|V| < 2^64 (e.g. 2^20 rows of values up to 2^43). A
// smaller threshold rescales often when the scores spread widely (fp8 rows whose
// group scales make a few rows score far above the rest).
constexpr float kRescaleLog2 = 64.0f;

struct Misc {
  uint64_t bar[kNumBars];
  uint32_t tmem_base;
  int abort;
  int progress;  // tiles whose stage fill has been issued (throttles the L2 prefetch warp)
  int pad0;
  float alpha[2][64];  // per stage: tile j+1 must not overwrite what tile j's rescale reads
  alignas(16) float inv[64];
  float lse2[64];
  uint8_t mask[2][8];  // sparse / gathered row validity per stage, one byte per 8 rows
};

template <int LAYOUT, bool TMA_KV>
struct Cfg {
  static constexpr int kNslab = (LAYOUT == 1) ? 8 : 9;
  static constexpr int kNope = (LAYOUT == 1) ? 448 : 512;
  static constexpr uint32_t kQBytes = kNslab * kSlab;
  static constexpr uint32_t kStageBytes = kNslab * kSlab;
  static constexpr uint32_t kOffStage = kQBytes;
  // P^T (64 query rows x 64 KV rows bf16) lives in the RoPE slab of its stage when
  // the row has 9 slabs (V only needs slabs 0-7); otherwise in two extra slabs.
  static constexpr bool kPInStage = (kNslab == 9);
  static constexpr uint32_t kOffP = kQBytes + 2 * kStageBytes;
  // fp8 rows carry group scales up to 2^k, so P is passed to the PV MMA as a bf16
  // pair P = P_hi + P_lo (P_lo = bf16(P - P_hi)) in extra 8 KB buffers: one per stage
  // where shared memory allows (8-slab rows), else one shared by both stages, whose
  // writer then waits for the previous tile's PV to finish.
  static constexpr bool kPSplit = (LAYOUT != 0);
  static constexpr uint32_t kOffPLo = kOffP + (kPInStage ? 0 : 2 * kSlab);
  static constexpr int kPLoBufs =
      !kPSplit ? 0 : (kOffPLo + 2 * kSlab + sizeof(Misc) + 1024 <= 232448 ? 2 : 1);
  static constexpr uint32_t kOffMisc = kOffPLo + kPLoBufs * kSlab;
  static constexpr uint32_t kSmem = kOffMisc + sizeof(Misc) + 1024;
  static_assert(kSmem <= 232448, "shared memory budget of one CTA");
  static constexpr int kChunks = (LAYOUT == 0) ? 72 : (kNope / 16 + 8);  // 16-B chunks per stored row
  static constexpr int kChunksPerThread = kChunks / 4;
  __device__ static uint32_t stage(uint32_t base, int st) { return base + kOffStage + st * kStageBytes; }
  __device__ static uint32_t parea(uint32_t base, int st) {
    return kPInStage ? stage(base, st) + 8 * kSlab : base + kOffP + st * kSlab;
  }
  __device__ static uint32_t plo(uint32_t base, int st) { return base + kOffPLo + (kPLoBufs == 2 ? st : 0) * kSlab; }
};

template <int LAYOUT, bool TMA_KV>
__global__ void __launch_bounds__(kDecodeThreads, 1)
    mla_decode_kernel(const __grid_constant__ DecodeParams P, const __grid_constant__ CUtensorMap q_map,
                      const __grid_constant__ CUtensorMap kv_map) {
  using C = Cfg<LAYOUT, TMA_KV>;
  constexpr int NS = C::kNslab;
  // Warp w runs on SM sub-partition w % 4 and reaches TMEM lanes 32 (w % 4) .. + 31, so
  // the four softmax warps 4-7 cover the four lane quarters of S and O^T. The PV issuer runs
  // on warp 3 and the L2 prefetch warp takes warp 1 (measured with the softmax on warps 4
  // and 5: DSV4-shaped decode 3 % faster, DSV3-shaped 0.5 %, verify 1.3 %). The sparse
  // variants keep the PV issuer on warp 1: their prefetch warp does per-row work and they
  // were 3 % slower.
  constexpr int kPvWarp = (LAYOUT == 1 || TMA_KV) ? 3 : 1;
  constexpr int kPrefetchWarp = (LAYOUT == 1 || TMA_KV) ? 1 : 3;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_addr(smem);
  Misc* misc = reinterpret_cast<Misc*>(smem + C::kOffMisc);
  auto bar = [&](int i) -> uint32_t { return smem_addr(&misc->bar[i]); };
  volatile int* abort_flag = &misc->abort;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // candidates listed per token: top-k positions (indices) or the rows of its slot runs
  // (gathered variants only: the TMA variant never sees either)
  const int32_t* const runs = TMA_KV ? nullptr : P.runs;
  const bool sparse = P.indices != nullptr || runs != nullptr;

  if (tid == 0) {
    mbar_init(bar(kQFull), 1);
    mbar_init(bar(kQEmpty), 1);
    for (int s = 0; s < 2; ++s) {
      for (int k = 0; k < 9; ++k) {
        // TMA path: one arrival (with its bytes) per slab of the group
        const int nslab_g = NS - 4 * k < 4 ? NS - 4 * k : 4;
        mbar_init(bar(kv_full(s, k)), TMA_KV ? (nslab_g > 0 ? nslab_g : 1) : 256);
      }
      for (int k = 0; k < 5; ++k) mbar_init(bar(kv_empty(s, k)), 1);
      mbar_init(bar(kSFull + s), 1);
      mbar_init(bar(kSFree + s), 128);
      mbar_init(bar(kPFull + s), 128);
    }
    mbar_init(bar(kPvDone), 1);
    mbar_init(bar(kOFull), 1);
    mbar_init(bar(kOFree), 128);
    mbar_init(bar(kFinal), 2);  // one commit from each MMA issuer
    misc->abort = 0;
    misc->progress = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&misc->tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The setup above overlaps the previous kernel's tail. Every role waits here for that
  // kernel before reading anything, except the L2 prefetch warp of the gathered variants:
  // it only reads tables to aim its hints (all lookups bounds-checked), and L2 is where the
  // previous kernel's writes land, so a line it warms early is still current when the other
  // roles read it after the wait. (Measured on the whole step: sparse 5 % and DSV4 0.5 %
  // faster; the bf16 TMA variant 2 % slower, its early hints queueing ahead of Q and the
  // first tiles, so it waits.)
  pdl_trigger();
  if (TMA_KV || warp != kPrefetchWarp) pdl_wait();
  const uint32_t tmem = misc->tmem_base;
  const uint32_t tmem_o = tmem;          // O^T: 4 blocks x 64 columns
  const uint32_t tmem_s = tmem + 256;    // S: 2 buffers x 64 columns

  const int G = P.groups;
  const int R = P.rows_per_req;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&q_map);
      if (TMA_KV) tma_prefetch_desc(&kv_map);
      int it = 0, u = 0;
      const int box_rows = P.page_size < kBlockRows ? P.page_size : kBlockRows;
      const int nbox = kBlockRows / box_rows;
      const uint32_t qbytes = NS * P.qbox_rows * 128;
      for (int w = blockIdx.x; w < P.num_work && !*abort_flag; w += gridDim.x) {
        const int part = w / G, g = w % G;
        for_each_unit(P, part, [&](int r, int lo, int hi, int) {
          if (*abort_flag) return;
          if (u > 0 && !mbar_wait(bar(kQEmpty), (u - 1) & 1, abort_flag, P.status)) return;
          mbar_arrive_expect_tx(bar(kQFull), qbytes);
          const int row0 = r * R + g * kGroupRows;
          for (int s = 0; s < NS; ++s) tma_load_2d(sb + s * kSlab, &q_map, s * 64, row0, bar(kQFull));
          ++u;
          if (!TMA_KV) {
            it += hi - lo;
            return;
          }
          const int L = P.seqlens[r];
          for (int j = lo; j < hi; ++j, ++it) {
            const int st = it & 1;
            int pages[8];  // page_size >= 8, so at most 64 / 8 boxes
            uint32_t bytes = 0;
            for (int k = 0; k < nbox; ++k) {
              const int pos0 = j * kBlockRows + k * box_rows;
              int page = -1;
              if (pos0 < L) {
                const int pi = pos0 >> P.log2_ps;
                page = pi < P.max_pages ? P.block_table[(int64_t)r * P.max_pages + pi] : -1;
                if (page < 0 || page >= P.num_pages) {
                  atomicOr(P.status, 2u);
                  page = -1;
                }
              }
              pages[k] = page;
              if (page >= 0) bytes += box_rows * 128;
            }
            const uint32_t dst = C::stage(sb, st);
            // slab by slab, each as soon as the PV that last read it has finished
            for (int s = 0; s < NS; ++s) {
              if (it >= 2 && (s == 8 || (s & 1) == 0) &&
                  !mbar_wait(bar(kv_empty(st, s == 8 ? 4 : s >> 1)), ((it >> 1) - 1) & 1, abort_flag, P.status))
                return;
              mbar_arrive_expect_tx(bar(kv_full(st, slab_group(s))), bytes);
              for (int k = 0; k < nbox; ++k) {
                if (pages[k] < 0) continue;
                const int in_page = (j * kBlockRows + k * box_rows) & (P.page_size - 1);
                tma_load_3d(dst + s * kSlab + k * box_rows * 128, &kv_map, s * 64, in_page, pages[k],
                            bar(kv_full(st, slab_group(s))));
              }
            }
            *reinterpret_cast<volatile int*>(&misc->progress) = it + 1;
          }
        });
      }
      // drain: wait for copies that may still be in flight after an abort
      if (*abort_flag) {
        if (u > 0) mbar_wait_drain(bar(kQFull), (u - 1) & 1);
        if (TMA_KV)
          for (int k = 1; k <= 2 && it - k >= 0; ++k)
            for (int gq = 0; gq <= slab_group(NS - 1); ++gq)
              mbar_wait_drain(bar(kv_full((it - k) & 1, gq)), ((it - k) >> 1) & 1);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ S issuer
    // (a compact rolled loop: it shares SMSP 2 with softmax warp 6 and converter warps,
    // whose large unrolled code would otherwise evict it from the instruction cache).
    // S and PV are issued by two threads: a thread that polls a barrier stalls
    // until the MMAs it has queued are dispatched, so a single issuer either
    // leaves the tensor pipe idle while it checks whether P is ready or issues
    // PV late. With two issuers, each waits only for its own operands and the
    // tensor pipe interleaves S(j+1) with PV(j) as soon as P(j) exists, which
    // frees each stage (and starts its refill) as early as possible.
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(64, 64, 0, 0);  // M = 64: rows over all four lane quarters
      const uint64_t kmaj = sdesc_sw128(0, 16, 1024);  // K-major: Q, K tile
      const uint64_t qa = kmaj | (sb >> 4);
      int it = 0, u = 0;
      for (int w = blockIdx.x; w < P.num_work && !*abort_flag; w += gridDim.x) {
        const int part = w / G;
        for_each_unit(P, part, [&](int, int lo, int hi, int) {
          if (*abort_flag) return;
          const int ntile = hi - lo;
          if (!mbar_wait(bar(kQFull), u & 1, abort_flag, P.status)) return;
          for (int jj = 0; jj < ntile; ++jj) {
            const int itj = it + jj;
            const int st = itj & 1;
            const uint32_t par = (itj >> 1) & 1;
            if (!TMA_KV && !mbar_wait(bar(kv_full(st, 0)), par, abort_flag, P.status)) return;
            if (itj >= 2 && !mbar_wait(bar(kSFree + st), par ^ 1u, abort_flag, P.status)) return;
            tc_fence_after();
            const uint32_t d = tmem_s + st * 64;
            uint64_t qs = qa, ksd = kmaj | (C::stage(sb, st) >> 4);
#pragma unroll 1
            for (int s = 0; s < NS; ++s) {
              if (TMA_KV && (s & 3) == 0 && !mbar_wait(bar(kv_full(st, slab_group(s))), par, abort_flag, P.status))
                return;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) mma_bf16_ss(d, qs + kk * 2, ksd + kk * 2, idesc_s, (s | kk) ? 1u : 0u);
              qs += kSlab >> 4;
              ksd += kSlab >> 4;
            }
            // (failure-detection test: withhold the first tile's signal so that the
            // softmax's bounded wait runs out)
            if (!(P.test_withhold_signal && itj == 0)) mma_commit(bar(kSFull + st));
          }
          mma_commit(bar(kQEmpty));
          it += ntile;
          ++u;
        });
      }
      // every MMA this thread issued must finish before TMEM is freed
      mma_commit(bar(kFinal));
      mbar_wait_drain(bar(kFinal), 0);
    }
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------ PV issuer
    // O^T += V^T P^T for each tile as soon as the softmax has written P^T(j)
    // (and, for a unit's first tile, the epilogue has read the previous O^T).
    if (lane == 0) {
      const uint64_t kmaj = sdesc_sw128(0, 16, 1024);     // K-major: P^T
      const uint64_t vmaj = sdesc_sw128(0, kSlab, 1024);  // MN-major: V^T (slab pairs)
      int it = 0, u = 0;
      for (int w = blockIdx.x; w < P.num_work && !*abort_flag; w += gridDim.x) {
        const int part = w / G, g = w % G;
        int rows_g = R - g * kGroupRows;
        rows_g = rows_g > kGroupRows ? kGroupRows : rows_g;
        const int nq = (rows_g + 15) & ~15;
        const uint32_t idesc_o = idesc_bf16_f32(128, nq, 1, 0);
        for_each_unit(P, part, [&](int, int lo, int hi, int) {
          if (*abort_flag) return;
          const int ntile = hi - lo;
          for (int jj = 0; jj < ntile; ++jj) {
            const int itj = it + jj;
            const int st = itj & 1;
            if (!mbar_wait(bar(kPFull + st), (itj >> 1) & 1, abort_flag, P.status)) return;
            if (jj == 0 && u > 0 && !mbar_wait(bar(kOFree), (u - 1) & 1, abort_flag, P.status)) return;
            tc_fence_after();
            const uint64_t pb = kmaj | (C::parea(sb, st) >> 4);
            const uint64_t plo = kmaj | (C::plo(sb, st) >> 4);
            // compact (rolled) issue loop: the issuing thread must not stall on instruction fetch
            uint64_t vblk = vmaj | (C::stage(sb, st) >> 4);
#pragma unroll 1
            for (int blk = 0; blk < 4; ++blk) {
              const uint32_t dcol = tmem_o + blk * 64;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(dcol, vblk + kk * (2048 >> 4), pb + kk * 2, idesc_o, (jj == 0 && kk == 0) ? 0u : 1u);
              if (C::kPSplit) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) mma_bf16_ss(dcol, vblk + kk * (2048 >> 4), plo + kk * 2, idesc_o, 1u);
              }
              mma_commit(bar(kv_empty(st, blk)));  // V slabs 2blk, 2blk+1 may be refilled
              vblk += (2 * kSlab) >> 4;
            }
            mma_commit(bar(kv_empty(st, 4)));
            mma_commit(bar(kPvDone));
          }
          mma_commit(bar(kOFull));
          it += ntile;
          ++u;
        });
      }
      mma_commit(bar(kFinal));
      mbar_wait_drain(bar(kFinal), 0);
    }
  } else if (warp == kPrefetchWarp) {
    // ------------------------------------------------------------ L2 prefetch
    // Streams the Q rows and KV rows of upcoming tiles from HBM into L2 so that
    // the stage fills (TMA or converters) find them there. It runs ahead of the
    // fills by about kPrefetchBytes and never blocks them: a prefetch is a hint.
    const int64_t tile_bytes = static_cast<int64_t>(kBlockRows) * (P.row_bytes + (LAYOUT != 0 ? 8 : 0));
    int ahead = static_cast<int>(kPrefetchBytes / tile_bytes);
    ahead = ahead < 2 ? 2 : ahead;
    const int box_rows = P.page_size < kBlockRows ? P.page_size : kBlockRows;
    const int nbox = kBlockRows / box_rows;
    const int64_t total_rows = static_cast<int64_t>(P.batch) * R;
    int pit = 0;
    for (int w = blockIdx.x; w < P.num_work && !*abort_flag; w += gridDim.x) {
      const int part = w / G, g = w % G;
      for_each_unit(P, part, [&](int r, int lo, int hi, int) {
        if (*abort_flag) return;
        if (lane == 0) {
          const int64_t row0 = static_cast<int64_t>(r) * R + g * kGroupRows;
          int64_t rows = total_rows - row0;
          rows = rows > P.qbox_rows ? P.qbox_rows : rows;
          if (rows > 0) prefetch_l2_bulk(P.q + row0 * (NS * 64), static_cast<uint32_t>(rows * NS * 64 * 2));
        }
        const int L = runs ? 0x7fffffff : request_len(P, r);
        const int tok = r * P.sq + (g * kGroupRows) / P.heads;
        const int4 rn = runs ? reinterpret_cast<const int4*>(runs)[tok] : make_int4(0, 0, 0, 0);
        for (int j = lo; j < hi; ++j, ++pit) {
          const uint64_t t0 = globaltimer();
          while (pit >= *reinterpret_cast<volatile int*>(&misc->progress) + ahead) {
            if (*abort_flag) return;
            if (globaltimer() - t0 > 20000000ull) break;  // stop throttling after 20 ms
            __nanosleep(256);
          }
          if (sparse && LAYOUT != 0 && !runs) {
            // fp8 rows gathered by top-k index get no L2 hints here (the converters hint each
            // row one tile ahead): measured on the sparse top-k workload (fp8-512), per-row hints
            // three tiles ahead raised DRAM traffic from 1.12x to 1.35x the algorithmic bytes
            // (rows evicted before their gather) and made the kernel 2 % slower. bf16 gathers
            // (sparse prefill: rows shared by many tokens) and window runs keep them (without:
            // 24 % and 3 % slower).
          } else if (sparse) {
            // two rows per lane: both indices, then both pages, then the prefetches
            int pos[2], page[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int kk = j * kBlockRows + lane + 32 * h;
              if (runs) pos[h] = kk < rn.w ? (kk < rn.y ? rn.x + kk : rn.z + kk - rn.y) : -1;
              else pos[h] = kk < P.topk ? P.indices[static_cast<int64_t>(tok) * P.topk + kk] : -1;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              page[h] = -1;
              if (pos[h] < 0 || pos[h] >= L) continue;
              const int pi = pos[h] >> P.log2_ps;
              // run slots (and positions of an unpaged run) are cache slots: page * page_size + offset
              if (runs || P.block_table == nullptr) page[h] = pi;
              else page[h] = pi < P.max_pages ? P.block_table[static_cast<int64_t>(r) * P.max_pages + pi] : -1;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (page[h] < 0 || page[h] >= P.num_pages) continue;
              const int off = pos[h] & (P.page_size - 1);
              const uint8_t* pg = P.kv + static_cast<int64_t>(page[h]) * P.page_bytes;
              prefetch_l2_bulk(pg + static_cast<int64_t>(off) * P.row_bytes, P.row_bytes);
              if (LAYOUT != 0) {
                const uintptr_t sa = reinterpret_cast<uintptr_t>(pg + static_cast<int64_t>(P.page_size) * P.row_bytes +
                                                                 off * 8);
                prefetch_l2_bulk(reinterpret_cast<const void*>(sa & ~uintptr_t(15)), 16);
              }
            }
          } else if (lane < nbox) {
            const int pos0 = j * kBlockRows + lane * box_rows;
            if (pos0 < L) {
              const int pi = pos0 >> P.log2_ps;
              const int page = pi < P.max_pages ? P.block_table[static_cast<int64_t>(r) * P.max_pages + pi] : -1;
              if (page >= 0 && page < P.num_pages) {
                const int rows = (L - pos0) < box_rows ? (L - pos0) : box_rows;
                const int off = pos0 & (P.page_size - 1);
                const uint8_t* pg = P.kv + static_cast<int64_t>(page) * P.page_bytes;
                prefetch_l2_bulk(pg + static_cast<int64_t>(off) * P.row_bytes,
                                 static_cast<uint32_t>(((rows * P.row_bytes) + 15) & ~15));
                if (LAYOUT != 0)
                  prefetch_l2_bulk(pg + static_cast<int64_t>(P.page_size) * P.row_bytes + off * 8,
                                   static_cast<uint32_t>((rows * 8 + 15) & ~15));
              }
            }
          }
        }
      });
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ softmax / epilogue
    // Warps 4-7 meet at named barriers (a waiting warp sleeps instead of taking
    // issue slots from the MMA issuers on the same SM sub-partitions). A named
    // barrier has no time limit, so these warps never leave one another behind:
    // a thread whose bounded wait fails only marks itself `dead` and carries on
    // through the barriers, every barrier ORs the mark in, and all four warps stop
    // together at the barrier where it becomes visible.
    const int wt = tid - 128;                 // 0..127, TMEM lane of this thread (O^T: value dims)
    const uint32_t lane_off = static_cast<uint32_t>((wt & ~31)) << 16;
    // S is an M = 64 accumulator: query row r at TMEM lane 32 (r / 16) + r % 16, so every warp
    // holds 16 rows, and the threads l and l + 16 of a warp take columns 0-31 and 32-63 of row
    // 16 w + l (they meet through shuffles)
    const int row = 16 * (wt >> 5) + (wt & 15);
    const int half = (wt >> 4) & 1;
    bool dead = false, stop = false;
    auto wait = [&](uint32_t b, uint32_t parity) {
      if (!dead && !mbar_wait(b, parity, abort_flag, P.status)) dead = true;
      return !dead;
    };
    int it = 0, u = 0;
    for (int w = blockIdx.x; w < P.num_work && !stop; w += gridDim.x) {
      const int part = w / G, g = w % G;
      int rows_g = R - g * kGroupRows;
      rows_g = rows_g > kGroupRows ? kGroupRows : rows_g;
      const int nq = (rows_g + 15) & ~15;
      for_each_unit(P, part, [&](int r, int lo, int hi, int sidx) {
        if (stop) return;
        const int L = runs ? 0x7fffffff : request_len(P, r);
        const int grow = g * kGroupRows + row;          // query row within the request
        const bool valid_row = row < rows_g;
        const int tok = grow / P.heads;
        int lim = L;
        if (P.causal && !sparse) {
          lim = L - P.sq + tok + 1;
          lim = lim > L ? L : lim;
        }
        float m_run = -INFINITY, l_run = 0.f;
        float m_true = -INFINITY;  // the largest scaled score (log2 units), for max_logits
        const int ntile = hi - lo;
        for (int jj = 0; jj < ntile; ++jj) {
          const int itj = it + jj;
          const int st = itj & 1;
          const int j = lo + jj;
          const bool first = jj == 0;
          bool need = false;
          {
            const uint32_t par = (itj >> 1) & 1;
            wait(bar(kSFull + st), par);
            if (!TMA_KV) wait(bar(kv_full(st, 0)), par);
          }
          // (a warp's two half-row threads exchange values below: a dead thread keeps going
          // through the shuffles with masked data and is stopped at the next barrier)
          {
            tc_fence_after();
            uint32_t sr[32];
            if (!dead) {
              tmem_ld16x2_32(tmem_s + st * 64 + lane_off, sr);
              tmem_wait_ld();
            }
            tc_fence_before();
            if (!dead) mbar_arrive(bar(kSFree + st));
            // mask (raw scores; the positive scale is folded into the exponent below)
            uint64_t vmask;
            if (sparse || !TMA_KV) {
              vmask = 0;
#pragma unroll
              for (int k = 0; k < 8; ++k) vmask |= static_cast<uint64_t>(misc->mask[st][k]) << (8 * k);
            }
            if (!sparse) {
              int nv = lim - j * kBlockRows;
              nv = nv < 0 ? 0 : (nv > 64 ? 64 : nv);
              vmask = nv == 64 ? ~0ull : ((1ull << nv) - 1ull);
            }
            if (!valid_row || dead) vmask = 0;
            const uint32_t hmask = static_cast<uint32_t>(vmask >> (32 * half));
            float x[32];
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              x[c] = ((hmask >> c) & 1u) ? __uint_as_float(sr[c]) : -INFINITY;
              m4[c & 3] = fmaxf(m4[c & 3], x[c]);
            }
            float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * P.scale_log2;
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));  // the row's maximum
            m_true = fmaxf(m_true, mt);
            const float m_new = (mt > m_run + kRescaleLog2) ? mt : m_run;
            need = (m_new != m_run) && (m_run != -INFINITY) && !first;
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = fast_exp2(m_run - m_use);
            float ps4[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t pk[16];
            uint32_t pl[C::kPSplit ? 16 : 1];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const float p0 = fast_exp2(fmaf(x[2 * c], P.scale_log2, -m_use));
              const float p1 = fast_exp2(fmaf(x[2 * c + 1], P.scale_log2, -m_use));
              ps4[c & 3] += p0 + p1;
              pk[c] = f32x2_to_bf16x2(p0, p1);
              if (C::kPSplit) {
                const float h0 = __uint_as_float(pk[c] << 16), h1 = __uint_as_float(pk[c] & 0xFFFF0000u);
                pl[c] = f32x2_to_bf16x2(p0 - h0, p1 - h1);
              }
            }
            l_run = l_run * alpha + ((ps4[0] + ps4[1]) + (ps4[2] + ps4[3]));  // this half's share
            m_run = m_new;
            if (half == 0) misc->alpha[st][row] = need ? alpha : 1.0f;
            // P^T row `row`: 64 bf16 along KV, K-major 128-B swizzled; this thread's 16-B chunks
            // are 4 half .. 4 half + 3
            const uint32_t pa = C::parea(sb, st) + row * 128;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              st_shared_v4(pa + (((4 * half + q4) ^ (row & 7)) << 4),
                           make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]));
            // a P_lo buffer of its own per stage is free as P_hi's is (the stage's tile two back
            // has completed its PV before this tile's rows were stored); a shared one once the
            // previous tile's PV has completed
            if (C::kPSplit && (C::kPLoBufs == 2 || itj == 0 || wait(bar(kPvDone), (itj - 1) & 1))) {
              const uint32_t pla = C::plo(sb, st) + row * 128;
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4)
                st_shared_v4(pla + (((4 * half + q4) ^ (row & 7)) << 4),
                             make_uint4(pl[4 * q4], pl[4 * q4 + 1], pl[4 * q4 + 2], pl[4 * q4 + 3]));
            }
          }
          if (TMA_KV && !sparse) {
            // rows past L in this tile may hold stale or non-finite bytes: zero their V part
            int nvalid = L - j * kBlockRows;
            nvalid = nvalid < 0 ? 0 : nvalid;
            if (nvalid < kBlockRows) {
              for (int gq = 0; gq < 2; ++gq) wait(bar(kv_full(st, gq)), (itj >> 1) & 1);
              if (!dead) {
                const uint32_t vs = C::stage(sb, st);
                const int nz = (kBlockRows - nvalid) * 8 * 8;  // rows x slabs x 16-B chunks
                for (int idx = wt; idx < nz; idx += 128) {
                  const int rr = nvalid + idx / 64;
                  const int sl = (idx / 8) & 7;
                  const int ch = idx & 7;
                  st_shared_v4(vs + sl * kSlab + rr * 128 + ch * 16, make_uint4(0, 0, 0, 0));
                }
              }
            }
          }
          fence_proxy_async_smem();
          // rescale needed anywhere, or a thread has given up (then everyone stops here)
          if (named_bar_or(1, 128, need || dead)) {
            if (named_bar_or(1, 128, dead)) {
              stop = true;
              return;
            }
            if (wait(bar(kPvDone), (itj - 1) & 1)) {
              tc_fence_after();
              // one TMEM round trip per 32 columns (columns past nq hold no query row)
              const float* al = misc->alpha[st];
#pragma unroll 1
              for (int k = 0; k < 8; ++k) {
                uint32_t t32[32];
                const uint32_t ta = tmem_o + lane_off + k * 32;
                tmem_ld32(ta, t32);
                tmem_wait_ld();
                const float* ak = al + (k & 1) * 32;
#pragma unroll
                for (int i = 0; i < 32; ++i) t32[i] = __float_as_uint(__uint_as_float(t32[i]) * ak[i]);
                tmem_st32(ta, t32);
              }
              tmem_wait_st();
              tc_fence_before();
            }
          }
          if (!dead) mbar_arrive(bar(kPFull + st));
        }
        // -------------------------------------------------------- epilogue
        const int base_split = P.num_splits[r];
        const int nsplit = P.num_splits[r + 1] - base_split;
        const int sg = base_split + sidx;
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 16);  // the row's sum over both halves
        if (half == 0) {
          float inv = 0.f, lse2 = -INFINITY;
          if (l_run > 0.f) {
            float denom = l_run;
            if (nsplit == 1 && P.sink != nullptr) {
              const int n = grow % P.heads;
              denom += fast_exp2(P.sink[n] * 1.4426950408889634f - m_run);
            }
            inv = 1.0f / denom;
            lse2 = m_run + log2f(l_run);
          }
          misc->inv[row] = inv;
          misc->lse2[row] = lse2;
          if (valid_row && !dead) {
            const float lse_nat = lse2 * 0.6931471805599453f;
            if (nsplit == 1) P.lse[(int64_t)r * R + grow] = lse_nat;
            else P.part_lse[(int64_t)sg * R + grow] = lse_nat;
            if (P.max_logits != nullptr) {
              const float mx = m_true * 0.6931471805599453f;  // back from log2 units: sm_scale * <q, k>
              if (nsplit == 1) P.max_logits[(int64_t)r * R + grow] = mx;
              else P.part_max[(int64_t)sg * R + grow] = mx;
            }
          }
        }
        if (named_bar_or(1, 128, dead)) {
          stop = true;
          return;
        }
        if (wait(bar(kOFull), u & 1)) {
          tc_fence_after();
          // row (query) qr of this unit goes to out[r * R + g * 64 + qr] (bf16) or to the
          // split partial part_out[sg * R + g * 64 + qr] (fp32); this thread writes value
          // dim blk * 128 + wt of each row, so consecutive rows are 512 elements apart
          const int64_t row0 = (nsplit == 1 ? (int64_t)r : (int64_t)sg) * R + g * kGroupRows;
          const float4* inv4 = reinterpret_cast<const float4*>(misc->inv);
          for (int blk = 0; blk < 4; ++blk) {
            const int d = blk * 128 + wt;
            for (int c = 0; c < nq; c += 16) {
              uint32_t t16[16];
              tmem_ld16(tmem_o + lane_off + blk * 64 + c, t16);
              float iv[16];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float4 f = inv4[(c >> 2) + k];
                iv[4 * k] = f.x;
                iv[4 * k + 1] = f.y;
                iv[4 * k + 2] = f.z;
                iv[4 * k + 3] = f.w;
              }
              tmem_wait_ld();
              const int nrow = rows_g - c < 16 ? rows_g - c : 16;
              if (nsplit == 1) {
                uint16_t* o = P.out + (row0 + c) * 512 + d;
                if (nrow == 16) {
#pragma unroll
                  for (int i = 0; i < 16; ++i)
                    o[i * 512] = static_cast<uint16_t>(f32x2_to_bf16x2(__uint_as_float(t16[i]) * iv[i], 0.f));
                } else {
#pragma unroll
                  for (int i = 0; i < 16; ++i)
                    if (i < nrow)
                      o[i * 512] = static_cast<uint16_t>(f32x2_to_bf16x2(__uint_as_float(t16[i]) * iv[i], 0.f));
                }
              } else {
                float* o = P.part_out + (row0 + c) * 512 + d;
                if (nrow == 16) {
#pragma unroll
                  for (int i = 0; i < 16; ++i) o[i * 512] = __uint_as_float(t16[i]) * iv[i];
                } else {
#pragma unroll
                  for (int i = 0; i < 16; ++i)
                    if (i < nrow) o[i * 512] = __uint_as_float(t16[i]) * iv[i];
                }
              }
            }
          }
          tc_fence_before();
          mbar_arrive(bar(kOFree));
        }
        it += ntile;
        ++u;
      });
    }
    // a thread that gave up after the last barrier of its last unit: nothing left to share
  } else if (warp >= 8 && !TMA_KV) {
    // ------------------------------------------------------------ converters
    const int ct = tid - 256;        // 0..255
    const int crow = ct >> 2;        // tile row handled
    const int part4 = ct & 3;        // chunk phase
    int it = 0;
    for (int w = blockIdx.x; w < P.num_work && !*abort_flag; w += gridDim.x) {
      const int part = w / G, g = w % G;
      for_each_unit(P, part, [&](int r, int lo, int hi, int) {
        if (*abort_flag) return;
        const int L = runs ? 0x7fffffff : request_len(P, r);
        const int tok = r * P.sq + (g * kGroupRows) / P.heads;   // sparse: the group's token
        const int4 rn = runs ? reinterpret_cast<const int4*>(runs)[tok] : make_int4(0, 0, 0, 0);
        // The address chain of a row (top-k index -> block_table entry -> row) runs two
        // tiles ahead of the conversion: the index of tile j + 2 and the page of tile j + 1
        // are loaded while tile j is converted, so only a unit's first tile waits for them.
        auto row_pos = [&](int j) -> int {  // KV position of this thread's row of tile j, or -1
          if (j >= hi) return -1;
          if (sparse) {
            const int kk = j * kBlockRows + crow;
            if (runs) return kk < rn.w ? (kk < rn.y ? rn.x + kk : rn.z + kk - rn.y) : -1;
            return kk < P.topk ? P.indices[(int64_t)tok * P.topk + kk] : -1;
          }
          return j * kBlockRows + crow;
        };
        auto row_page = [&](int pos) -> int {  // its page; -1 if no row, -2 if the entry is bad
          if (pos < 0 || pos >= L) return -1;
          const int pi = pos >> P.log2_ps;
          // run slots (and positions of an unpaged run) are cache slots (page * page_size +
          // offset), not positions of the request
          const int page = (runs || P.block_table == nullptr)
                               ? pi
                               : (pi < P.max_pages ? P.block_table[(int64_t)r * P.max_pages + pi] : -1);
          return (page < 0 || page >= P.num_pages) ? -2 : page;
        };
        int pos_a = row_pos(lo), pos_b = row_pos(lo + 1);
        int page_a = row_page(pos_a);
        for (int j = lo; j < hi; ++j, ++it) {
          const int st = it & 1;
          const int pos = pos_a, page = page_a;
          pos_a = pos_b;
          page_a = row_page(pos_b);
          pos_b = row_pos(j + 2);
          if (sparse && LAYOUT != 0 && !runs && page_a >= 0) {
            // L2 hints for this thread's share of its row of the next tile: one tile ahead, the
            // distance at which the hinted rows are still in L2 when gathered (the prefetch warp
            // gives these rows none; measured on the sparse top-k workload: 2 % faster)
            const int offn = pos_a & (P.page_size - 1);
            const uint8_t* pgn = P.kv + (int64_t)page_a * P.page_bytes;
            const uint8_t* rn = pgn + (int64_t)offn * P.row_bytes;
            for (int l = part4; l * 128 < P.row_bytes; l += 4) prefetch_l2_line(rn + l * 128);
            if (part4 == 3) prefetch_l2_line(pgn + (int64_t)P.page_size * P.row_bytes + offn * 8);
          }
          bool valid = page >= 0;
          if (page == -2 && part4 == 0) atomicOr(P.status, 2u);
          const uint8_t* rowp = nullptr;
          const uint8_t* scp = nullptr;
          if (valid) {
            const int off = pos & (P.page_size - 1);
            rowp = P.kv + (int64_t)page * P.page_bytes + (int64_t)off * P.row_bytes;
            scp = P.kv + (int64_t)page * P.page_bytes + (int64_t)P.page_size * P.row_bytes + off * 8;
          }
          const unsigned bal = __ballot_sync(0xffffffffu, valid && part4 == 0);
          // issue this tile's global loads first, then wait for the stage to be free
          constexpr int CPT = C::kChunksPerThread;
          uint4 v[CPT];
#pragma unroll
          for (int i = 0; i < CPT; ++i) {
            const int c = part4 + 4 * i;
            v[i] = valid ? ld_nc_v4(rowp + c * 16) : make_uint4(0, 0, 0, 0);
          }
          uint2 sc = make_uint2(0, 0);
          if (LAYOUT != 0 && valid) sc = ld_nc_v2(scp);
          // dequantise in registers before waiting for the stage, so that only the stores
          // remain once the PV two tiles back has released it: an fp8 chunk (16 e4m3 codes of
          // group c/4) becomes 16 bf16 in lo/hi; a bf16 (RoPE) chunk stays in lo
          uint4 lo[CPT], hi[CPT];
#pragma unroll
          for (int i = 0; i < CPT; ++i) {
            const int c = part4 + 4 * i;
            lo[i] = v[i];
            hi[i] = make_uint4(0, 0, 0, 0);
            if (LAYOUT != 0 && c < C::kNope / 16) {
              const int grp = c >> 2;
              const uint32_t sbyte = (grp < 4 ? (sc.x >> (8 * grp)) : (sc.y >> (8 * (grp - 4)))) & 0xFFu;
              const float scale = valid ? ue8m0_to_f32(sbyte) : 0.f;
              const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
              uint32_t o[8];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float2 a = e4m3x2_to_f32x2(w4[q] & 0xFFFFu);
                const float2 b = e4m3x2_to_f32x2(w4[q] >> 16);
                o[2 * q] = f32x2_to_bf16x2(a.x * scale, a.y * scale);
                o[2 * q + 1] = f32x2_to_bf16x2(b.x * scale, b.y * scale);
              }
              lo[i] = make_uint4(o[0], o[1], o[2], o[3]);
              hi[i] = make_uint4(o[4], o[5], o[6], o[7]);
            }
          }
          if (it >= 2 && !mbar_wait(bar(kv_empty(st, 4)), ((it >> 1) - 1) & 1, abort_flag, P.status)) return;
          fence_proxy_async_smem();
          if (lane == 0) {
            uint32_t byte = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) byte |= ((bal >> (4 * k)) & 1u) << k;
            misc->mask[st][(ct >> 5)] = static_cast<uint8_t>(byte);
          }
          const uint32_t dst = C::stage(sb, st);
#pragma unroll
          for (int i = 0; i < CPT; ++i) {
            const int c = part4 + 4 * i;
            if (LAYOUT == 0) {
              // bf16 copy: chunk c = dims [8c, 8c + 8)
              st_shared_v4(dst + (c >> 3) * kSlab + sw128_offset(crow, (c & 7) * 8), lo[i]);
            } else if (c < C::kNope / 16) {
              // dims [16c, 16c + 16) of slab c/4
              const uint32_t sl = dst + (c >> 2) * kSlab;
              const int k0 = (c & 3) * 16;
              st_shared_v4(sl + sw128_offset(crow, k0), lo[i]);
              st_shared_v4(sl + sw128_offset(crow, k0 + 8), hi[i]);
            } else {
              // RoPE: 8 bf16 at dims [nope + 8k, nope + 8k + 8)
              const int dim = C::kNope + 8 * (c - C::kNope / 16);
              st_shared_v4(dst + (dim >> 6) * kSlab + sw128_offset(crow, dim & 63), lo[i]);
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(bar(kv_full(st, 0)));
          if (ct == 0) *reinterpret_cast<volatile int*>(&misc->progress) = it + 1;
        }
      });
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

size_t decode_smem_bytes(DecodeVariant v) {
  switch (v) {
    case DecodeVariant::kBf16Tma: return Cfg<0, true>::kSmem;
    case DecodeVariant::kBf16Gather: return Cfg<0, false>::kSmem;
    case DecodeVariant::kFp8_448: return Cfg<1, false>::kSmem;
    case DecodeVariant::kFp8_512: return Cfg<2, false>::kSmem;
  }
  return 0;
}

template <int LAYOUT, bool TMA_KV>
static cudaError_t launch_variant(const DecodeParams& p, const CUtensorMap& q_map, const CUtensorMap& kv_map, int grid,
                                  cudaStream_t stream) {
  auto kern = mla_decode_kernel<LAYOUT, TMA_KV>;
  const size_t smem = Cfg<LAYOUT, TMA_KV>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(kDecodeThreads), smem, stream, p, q_map, kv_map);
}

cudaError_t launch_decode(DecodeVariant v, const DecodeParams& p, const CUtensorMap& q_map, const CUtensorMap& kv_map,
                          int grid, cudaStream_t stream) {
  switch (v) {
    case DecodeVariant::kBf16Tma: return launch_variant<0, true>(p, q_map, kv_map, grid, stream);
    case DecodeVariant::kBf16Gather: return launch_variant<0, false>(p, q_map, kv_map, grid, stream);
    case DecodeVariant::kFp8_448: return launch_variant<1, false>(p, q_map, kv_map, grid, stream);
    case DecodeVariant::kFp8_512: return launch_variant<2, false>(p, q_map, kv_map, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace mla
