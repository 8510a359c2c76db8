// Implicit-GEMM conv2d + BatchNorm + SiLU on the 5th-generation tensor cores.
//
// GEMM view: M = N*Ho*Wo output pixels, N_gemm = C_out, K = KH*KW*C_in in
// (kh, kw, ci) order, which is the channels-last (OHWI) filter layout
// ("When the fusion you want is impossible, fuse into the producer": the
// filters are packed channels-last once at load time).  The A operand is never
// materialised: TMA's im2col mode gathers 128 output pixels x 64 channels of
// the NHWC input for one filter tap straight into shared memory (zero fill at
// the padding), which is the TMA_LOAD_IM2COL -> UMMA path that page describes;
// a 1x1 stride-1 unpadded convolution is a plain matrix, loaded as a 2-D tile.
// A CTA's tile is 128 output pixels, or 256 (wide tiles: two 128-row MMAs per
// K step on one B stage).
//
// Persistent kernel, one CTA (or, with CL = 2, one CTA pair) per SM, with
// 2 + EPI warps:
//   warp 0  TMA producer: a ring of up to 6 shared-memory stages sized by the
//           host's shared-memory plan (A 16 KB + B BN*128 B per stage, or A
//           alone when the filter block is resident)
//   warp 1  TMEM allocator and MMA issuer: tcgen05.mma M=128, N=BN, K=16, fp32
//           accumulators in TMEM, double-buffered so the epilogue of one tile
//           overlaps the main loop of the next (single for the 256 x 256
//           accumulator of a wide tile, which fills TMEM)
//   warps 2.. epilogue ("Fusing an Epilogue", "The shape of it"), 16 warps for
//           short K loops and 8 for long ones: TMEM -> registers,
//           v = acc*scale[co] + bias[co], v*sigmoid(v), bf16, then a swizzled
//           shared-memory box and a TMA store.  The per-channel parameters are
//           read inside the kernel, as in the page's BatchNorm-epilog listing.
// Every mbarrier wait is bounded (see ptx::mbar_wait); a role that times out
// sets the device error word and winds down, and the CTA drains its in-flight
// copies and MMAs before it frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <string.h>

#include "ptx_sm100.cuh"
#include "tf_internal.h"

namespace tf {
namespace {

constexpr int BM = 128;            // output pixels per tile (UMMA M)
constexpr int BK = 64;             // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int UMMA_K = 16;
constexpr int kMaxStages = 8;      // deepest operand ring the shared-memory plan may choose
constexpr int kMaxStagesStreamed = 6;   // ... when B streams through the ring with A
constexpr int kSmemLimit = 227 * 1024;        // opt-in dynamic shared memory per block
constexpr int kBResMaxBytes = 128 * 1024;     // largest filter block kept resident in shared memory
constexpr int kParamChunkBytes = 64 * 4;      // 32 scale + 32 bias floats of one 32-channel chunk
// Epilogue warps: 16 (four per TMEM lane quarter) for short K loops, where the
// epilogue paces the kernel; 8 for long ones, where it hides behind the MMAs.
constexpr int kEpiWarpsShortK = 16, kEpiWarpsLongK = 8;
constexpr int threads_for(int epi_warps) { return 64 + 32 * epi_warps; }
// 32-channel accumulator chunks each epilogue warp handles per tile
constexpr int chunks_per_warp(int bn, int epi_warps) { return bn / 32 / (epi_warps / 4) > 0 ? bn / 32 / (epi_warps / 4) : 1; }
constexpr int kOutBox = 32;        // epilogue store box: 32 pixels x 32 channels (64 B rows)
constexpr int kOutBoxBytes = kOutBox * kOutBox * 2;

constexpr int kABytes = BM * BK * 2;          // one A (im2col) tile of a K step
constexpr int kNumBars = 2 * kMaxStages + 5;  // full, empty, tmem full x2, tmem empty x2, drain
constexpr int kBarBytes = kNumBars * 8 + 16;  // + the TMEM address slot

// MH: 128-row halves per CTA tile (1, or 2 for 256-row tiles whose two MMAs
// per K step share one B stage).  The fp32 accumulator of a tile takes MH*BN
// TMEM columns; two of them (double buffering) when they fit in the 512.
template <int BN, int MH = 1, int CG = 1>
struct Tile {
    static constexpr int B_BYTES = BN * BK * 2 / CG;   // this CTA's share of a K step's B (filter) tile
    static constexpr int NACC = 2 * MH * BN <= 512 ? 2 : 1;
    static constexpr uint32_t TMEM_COLS = NACC * MH * BN < 32 ? 32 : NACC * MH * BN;
};

// Shared-memory plan, from the 1024-byte-aligned base (operand tiles use
// the 128-byte swizzle, whose atoms are 1024 B):
//   [0, off_bres)          operand ring: `stages` x (A tile, + B tile unless resident)
//   [off_bres, off_out)    resident filter block: num_kb B tiles (b_res only)
//   [off_out, off_par)     one 2 KB output staging box per epilogue warp
//   [off_par, off_bar)     per epilogue warp, the scale/bias values of its chunks;
//                          with a resident filter block (whose channel tile never
//                          changes) one table of the tile's BN scales and biases
//   [off_bar, total)       mbarriers and the TMEM address slot
struct SmemPlan {
    int stages, stage_bytes, b_res, off_bres, off_out, off_par, off_bar, alloc;
};

struct UmmaParams {
    const float *scale;
    const float *bias;
    __nv_bfloat16 *y;
    uint32_t *err;
    uint64_t wait_ns;
    int M, C_out, KW, HoWo, Wo;
    int m_base;              // first output row of this launch's tiles (a wide kernel's tail launch)
    int stride_h, stride_w, pad_h, pad_w;
    int num_kb, cblocks, num_n_tiles, num_tiles;
    int epilogue;            // 0: plain bf16 store, 1: BN + SiLU, 2: fp32 split-K partial to ws
    int y_direct;            // 1: rows of y are not a multiple of 16 bytes (C_out % 8 != 0), so no
                             // TMA store: each warp copies its staging box to y with masked stores
    int splits, kb_per_split, num_work;   // work item = (tile, K split), split fastest
    // Items from split_from on are parts of tiles (BN/parts channels each):
    // item split_from + parts*i + j is part j of tile split_from + i.  Only
    // with a resident filter block, one channel tile and one K split, so that
    // the last, partial wave of tiles is spread over `parts` times the CTAs.
    int split_from, parts;
    float *ws;               // split-K partials [splits][M][C_out] (epilogue 2 only)
    SmemPlan sm;
};

// CL: CTAs per cluster along M (1 or 2).  With CL = 2 the two CTAs of a
// cluster take vertically adjacent output tiles that read the same filter
// (B) tile at the same time, so the second read of each B tile is an L2 hit
// on the same GPC; each CTA loads its own operands and the two share nothing
// else (no cross-CTA copies or barriers in the pipeline).
//
// Resident filter (p.sm.b_res, one K split only): when the whole [K][BN]
// filter block of the CTA's output-channel tile fits in shared memory (K <=
// 256 at BN = 256: a 1x1 convolution of up to 256 input channels; with a
// paired MMA each CTA holds only its half of the block, so up to 512) it is
// loaded once, K step by K step alongside the A tiles of the CTA's first
// tile, and afterwards only A streams through the ring: a memory-bound
// convolution then moves just its activations and outputs through each SM
// instead of re-reading the filters from L2 for every tile, and the ring can
// be deeper.  The host launches a multiple of num_n_tiles CTAs (or pairs), so
// that each keeps one channel tile.
//
// Wide tiles (MH = 2): each CTA's tile is 256 output pixels, two 128-row
// MMAs per K step reading the same B stage, so every SM moves 64 KB of
// operands per 1024 tensor cycles instead of 48 KB per 512.  Their 256 x BN
// accumulator fills TMEM at BN = 256, so it is single-buffered: the MMAs of a
// tile wait for the epilogue of the previous one, a short pause against a
// long K loop.  A last, partial wave of at most half the units goes to a
// second launch on 128-row tiles (leave_wide_tail); where no full wave
// precedes it, items from split_from on are instead the 128-row halves of
// its tiles (parts = 2) in this launch.
//
// Paired MMA (CG = 2, on CL = 2 clusters): the two CTAs of a pair run one
// tcgen05.mma.cta_group::2 of M = 256 (128 rows per CTA, MH of them per K
// step) issued by the first CTA.  Each CTA loads its own A rows and HALF of
// the filter tile (BN/2 rows), and the tensor cores of both SMs read both
// halves: the pair shares B without any copy between the CTAs.  Every SM then
// moves 16 KB of A + BN*64 B of B per 64-deep K step (BN = 256: 32 KB per
// 512 tensor cycles), and its accumulator is 128 x BN, so at BN = 256 two of
// them still fit in TMEM (double buffering).  Both CTAs' copies complete on
// the first CTA's `full` barrier (.cta_group::2 loads), the first CTA's MMA
// commits release the stages and hand over the accumulators in both CTAs,
// and both CTAs' epilogue warps report a drained accumulator to the first
// CTA's `tempty` barrier.
template <int BN, bool IM2COL, int CL, int kEpiWarps, int MH = 1, int CG = 1>
__global__ void __launch_bounds__(threads_for(kEpiWarps), 1)
    conv_umma_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                     const __grid_constant__ CUtensorMap tmap_y, const UmmaParams p)
{
    static_assert(CG == 1 || CL == 2, "a paired MMA runs on a 2-CTA cluster");
    constexpr bool PAIR = CG == 2;
    using T = Tile<BN, MH, CG>;
    // operand tiles use the 128-byte swizzle, whose 8-row atoms must start on
    // 1024-byte boundaries (checked below)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.sm.off_bar);
    uint64_t *empty = full + kMaxStages;
    uint64_t *tfull = empty + kMaxStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    const int nstages = p.sm.stages;
    const bool b_res = p.sm.b_res != 0;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int crank = CL > 1 ? (int)ptx::cluster_ctarank() : 0;
    const int cid = (int)blockIdx.x / CL, ncl = (int)gridDim.x / CL;   // cluster index and count
    const bool leader = !PAIR || crank == 0;   // the CTA whose thread issues the (paired) MMAs

    if (threadIdx.x == 0) {
        for (int s = 0; s < nstages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);    // released by this CTA's MMA thread
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&tfull[b], 1);
            // every epilogue thread arrives; with a paired MMA, one lane per
            // epilogue warp of either CTA arrives on the first CTA's barrier
            ptx::mbar_init(&tempty[b], PAIR ? 2 * kEpiWarps : kEpiWarps * 32);
        }
        ptx::mbar_init(drain, 1);
        ptx::mbar_init_fence();
        ptx::prefetch_tensormap(&tmap_a);
        ptx::prefetch_tensormap(&tmap_b);
        if (!p.y_direct) ptx::prefetch_tensormap(&tmap_y);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            ptx::tmem_alloc_pair(tmem_slot, T::TMEM_COLS);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(tmem_slot, T::TMEM_COLS);
            ptx::tmem_relinquish();
        }
    }
    ptx::tc_fence_before();
    cta_sync();
    ptx::tc_fence_after();
    // a pair's barriers exist in both CTAs before any copy, commit or arrival
    // from the other CTA reaches them
    if constexpr (PAIR) ptx::cluster_sync();
    // Programmatic dependent launch: the next kernel of the stream may start
    // its own set-up on SMs this grid leaves.  Each role waits for the
    // stream's previous kernel (griddep_wait) only right before its first
    // global-memory access, so that the set-up above and the first work
    // item's address arithmetic overlap that kernel's tail.
    ptx::griddep_launch_dependents();
    const uint32_t tmem_base = *tmem_slot;
    int num_work = p.num_work;
    if ((ptx::smem_u32(smem) & 1023u) != 0) {   // no work on misaligned operand tiles
        num_work = 0;
        if (threadIdx.x == 0) atomicOr(p.err, TF_DEVERR_SMEM_ALIGN);
    }
    if constexpr (PAIR) {
        // the paired MMA writes both CTAs' accumulators at the first CTA's
        // TMEM address: if the two allocations differ, no work is done
        if (ptx::ld_shared_cluster_u32(ptx::mapa_shared(tmem_slot, (uint32_t)crank ^ 1u)) != tmem_base) {
            num_work = 0;
            if (threadIdx.x == 0) atomicOr(p.err, TF_DEVERR_PAIR_TMEM);   // an OR: order-free
        }
    }

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, last_phase = 0;  // per-stage bit masks
            bool ok = true, waited = false;
            for (int work = cid; ok && work < num_work; work += ncl) {
                // a resident filter block streams in with the CTA's first tile:
                // K step kb's B tile lands in its resident slot on the same
                // barrier as that step's A tile
                const bool first = work == cid;
                const int part = work < p.split_from ? -1 : (work - p.split_from) % p.parts;
                const int tile = work < p.split_from ? work / p.splits
                                                     : p.split_from + (work - p.split_from) / p.parts;
                const int kb_begin = work < p.split_from ? (work - tile * p.splits) * p.kb_per_split : 0;
                const int kb_end = min(kb_begin + p.kb_per_split, p.num_kb);
                const int mh = MH > 1 && part >= 0 ? 1 : MH;   // 128-row halves this item loads
                const int m0 = p.m_base + ((tile / p.num_n_tiles) * CL + crank) * (BM * MH) +
                               (MH > 1 && part > 0 ? part * BM : 0);
                const int n0 = (tile % p.num_n_tiles) * BN;
                int img[MH], w_base[MH], h_base[MH];
#pragma unroll
                for (int hh = 0; hh < MH; ++hh) {
                    const int mr = m0 + hh * BM;
                    img[hh] = mr / p.HoWo;
                    const int rem = mr - img[hh] * p.HoWo;
                    const int oh = rem / p.Wo, ow = rem - (rem / p.Wo) * p.Wo;
                    w_base[hh] = ow * p.stride_w - p.pad_w;
                    h_base[hh] = oh * p.stride_h - p.pad_h;
                }
                for (int kb = kb_begin; kb < kb_end; ++kb) {
                    if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    if (!waited) {   // the first copy reads memory the previous kernel may write
                        ptx::griddep_wait();
                        waited = true;
                    }
                    // bytes this CTA loads for the stage; with a paired MMA both CTAs
                    // load as much, and all of it completes on the first CTA's barrier
                    const uint32_t own = (uint32_t)(p.sm.stage_bytes - (MH - mh) * kABytes +
                                                    (b_res && first ? T::B_BYTES : 0));
                    if (leader) ptx::mbar_arrive_expect_tx(&full[stage], PAIR ? 2 * own : own);
                    const uint32_t full_pair = PAIR ? ptx::mapa_shared(&full[stage], 0) : 0u;
                    uint8_t *a_dst = smem + stage * p.sm.stage_bytes;
                    uint8_t *b_dst = a_dst + MH * kABytes;
                    const int tap = kb / p.cblocks;
                    const int c0 = (kb - tap * p.cblocks) * BK;
                    for (int hh = 0; hh < mh; ++hh) {
                        if constexpr (IM2COL) {
                            const int kh = tap / p.KW, kw = tap - (tap / p.KW) * p.KW;
                            if constexpr (PAIR)
                                ptx::tma_load_im2col_4d_pair(a_dst + hh * kABytes, &tmap_a, full_pair, c0,
                                                             w_base[hh], h_base[hh], img[hh], (uint16_t)kw,
                                                             (uint16_t)kh);
                            else
                                ptx::tma_load_im2col_4d(a_dst + hh * kABytes, &tmap_a, &full[stage], c0,
                                                        w_base[hh], h_base[hh], img[hh], (uint16_t)kw,
                                                        (uint16_t)kh);
                        } else {
                            // rows past M are never stored: a box lying wholly past M (the second
                            // CTA of a pair, a wide tile's half) starts at the last row instead, so
                            // that every tiled load overlaps the tensor
                            const int row = min(m0 + hh * BM, p.M - 1);
                            if constexpr (PAIR)
                                ptx::tma_load_2d_pair(a_dst + hh * kABytes, &tmap_a, full_pair, c0, row);
                            else
                                ptx::tma_load_2d(a_dst + hh * kABytes, &tmap_a, &full[stage], c0, row);
                        }
                    }
                    // B: filter tap `tap`, input channels c0 .. c0+63 (zero past C_in), BN
                    // output channels (zero past C_out) -- or this CTA's half of them
                    if constexpr (PAIR) {
                        if (!b_res)
                            ptx::tma_load_3d_pair(b_dst, &tmap_b, full_pair, c0, tap, n0 + crank * (BN / 2));
                        else if (first)
                            ptx::tma_load_3d_pair(smem + p.sm.off_bres + kb * T::B_BYTES, &tmap_b, full_pair, c0,
                                                  tap, n0 + crank * (BN / 2));
                    } else if (!b_res)
                        ptx::tma_load_3d(b_dst, &tmap_b, &full[stage], c0, tap, n0);
                    else if (first)
                        ptx::tma_load_3d(smem + p.sm.off_bres + kb * T::B_BYTES, &tmap_b, &full[stage], c0, tap, n0);
                    issued |= 1u << stage;
                    last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == nstages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) atomicOr(p.err, TF_DEVERR_PRODUCER_WAIT);
            // Every issued copy must have landed before the CTA may exit (a
            // pair's copies all complete on the first CTA's barriers, which its
            // producer drains before the pair's closing cluster barrier).
            for (int s = 0; s < nstages; ++s)
                if (leader && ((issued >> s) & 1u))
                    if (!ptx::mbar_wait(&full[s], (last_phase >> s) & 1u, p.wait_ns))
                        atomicOr(p.err, TF_DEVERR_DRAIN_WAIT);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && leader) {
            ptx::griddep_wait();   // (its only global access is the error word)
            constexpr uint32_t idesc = ptx::idesc_bf16_f32(PAIR ? 2 * BM : BM, BN);
            constexpr uint32_t idesc_half = ptx::idesc_bf16_f32(PAIR ? 2 * BM : BM, BN / 2);
            constexpr uint32_t idesc_quarter = ptx::idesc_bf16_f32(PAIR ? 2 * BM : BM, BN / 4);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int local = 0;
            for (int work = cid; ok && work < num_work; work += ncl, ++local) {
                const int kb_begin = work < p.split_from ? (work % p.splits) * p.kb_per_split : 0;
                const int kb_end = min(kb_begin + p.kb_per_split, p.num_kb);
                // part j of a tile: N = BN/parts on rows [j*BN/parts, +BN/parts) of the resident block
                // (MH = 1; with a paired MMA, rows [j*BN/parts/2, +BN/parts/2) of each CTA's half of
                // it), or its 128-row half j (MH = 2)
                const int part = work < p.split_from ? -1 : (work - p.split_from) % p.parts;
                const int mh = MH > 1 && part >= 0 ? 1 : MH;
                const uint32_t id = MH > 1 || part < 0 ? idesc : (p.parts == 2 ? idesc_half : idesc_quarter);
                const uint32_t b_half = MH == 1 && part > 0 ? (uint32_t)(part * (BN / p.parts / CG)) * (BK * 2) : 0u;
                const int b = T::NACC == 2 ? local & 1 : 0;
                const uint32_t acc_phase = T::NACC == 2 ? (uint32_t)(local >> 1) & 1u : (uint32_t)local & 1u;
                // (cluster-scope acquire for a pair: the peer's epilogue arrives here)
                if (!ptx::mbar_wait<PAIR>(&tempty[b], acc_phase ^ 1u, p.wait_ns)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(b * MH * BN);
                for (int kb = kb_begin; kb < kb_end; ++kb) {
                    if (!ptx::mbar_wait(&full[stage], phase, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a_addr = ptx::smem_u32(smem + stage * p.sm.stage_bytes);
                    const uint32_t b_addr = b_res ? ptx::smem_u32(smem + p.sm.off_bres + kb * T::B_BYTES) + b_half
                                                  : a_addr + MH * kABytes;
                    for (int hh = 0; hh < mh; ++hh) {
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k) {
                            const uint64_t ad = ptx::sw128_kmajor_desc(a_addr + hh * kABytes + k * UMMA_K * 2);
                            const uint64_t bd = ptx::sw128_kmajor_desc(b_addr + k * UMMA_K * 2);
                            const uint32_t acc = (kb > kb_begin || k > 0) ? 1u : 0u;
                            if constexpr (PAIR)
                                ptx::umma_bf16_pair(d_tmem + (uint32_t)(hh * BN), ad, bd, id, acc);
                            else
                                ptx::umma_bf16(d_tmem + (uint32_t)(hh * BN), ad, bd, id, acc);
                        }
                    }
                    // frees the stage (in both CTAs of a pair) once these MMAs have read it
                    if constexpr (PAIR) {
                        ptx::umma_commit_pair(ptx::mapa_shared(&empty[stage], 0));
                        ptx::umma_commit_pair(ptx::mapa_shared(&empty[stage], 1));
                    } else {
                        ptx::umma_commit(&empty[stage]);
                    }
                    if (++stage == nstages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                // accumulator complete (in both CTAs of a pair)
                if constexpr (PAIR) {
                    ptx::umma_commit_pair(ptx::mapa_shared(&tfull[b], 0));
                    ptx::umma_commit_pair(ptx::mapa_shared(&tfull[b], 1));
                } else {
                    ptx::umma_commit(&tfull[b]);
                }
            }
            if (!ok) atomicOr(p.err, TF_DEVERR_MMA_WAIT);
            if constexpr (PAIR)
                ptx::umma_commit_pair(ptx::smem_u32(drain));
            else
                ptx::umma_commit(drain);
            if (!ptx::mbar_wait(drain, 0, p.wait_ns)) atomicOr(p.err, TF_DEVERR_DRAIN_WAIT);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Warp w reads TMEM lanes 32*(w%4) .. +31 (one output pixel per lane)
        // and the 32-column chunks c = h, h+4, ... of the accumulator.  Each
        // chunk becomes 32 pixels x 32 channels of bf16 in a 64-byte-swizzled
        // staging box, written to y by one TMA store.  Sixteen warps (four per
        // SM sub-partition) keep the special-function and FMA pipes busy
        // while others wait on TMEM loads and stores.  Every lane needs all 32
        // scale and bias values of a chunk: the warp keeps those of its chunks
        // in a shared-memory slice (one coalesced load per lane and chunk,
        // repeated only when the tile's channel range changes) and reads them
        // with broadcast loads.
        ptx::griddep_wait();   // before the parameter and output accesses
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        uint8_t *box = smem + p.sm.off_out + (warp - 2) * kOutBoxBytes;
        constexpr int kChunks = chunks_per_warp(BN, kEpiWarps);
        float *slice = reinterpret_cast<float *>(smem + p.sm.off_par + (warp - 2) * kChunks * kParamChunkBytes);
        // A resident filter block pins the CTA to one channel tile: its BN
        // scales and biases are loaded once into a table all epilogue warps read.
        float *table = reinterpret_cast<float *>(smem + p.sm.off_par);
        const int cta_n0 = (cid % p.num_n_tiles) * BN;
        if (b_res && p.epilogue == 1) {
            for (int i = threadIdx.x - 64; i < BN; i += kEpiWarps * 32) {
                const bool in = cta_n0 + i < p.C_out;
                table[i] = in ? __ldg(p.scale + cta_n0 + i) : 0.0f;
                table[BN + i] = in ? __ldg(p.bias + cta_n0 + i) : 0.0f;
            }
            __syncwarp();
            asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");   // the epilogue warps only
        }
        int slice_n0 = -1;   // 8 * first channel + parts of the item whose parameters the slice holds
        int local = 0;
        bool ok = true;
        for (int work = cid; work < num_work; work += ncl, ++local) {
            const int part = work < p.split_from ? -1 : (work - p.split_from) % p.parts;
            const int tile = part < 0 ? work / p.splits : p.split_from + (work - p.split_from) / p.parts;
            const int split = part < 0 ? work - tile * p.splits : 0;
            const bool npart = MH == 1 && part >= 0;          // a part along the channels
            const int mh = MH > 1 && part >= 0 ? 1 : MH;     // 128-row halves of this item
            const int width = npart ? BN / p.parts : BN;       // channels of this item
            const int m0 = p.m_base + ((tile / p.num_n_tiles) * CL + crank) * (BM * MH) +
                           (MH > 1 && part > 0 ? part * BM : 0);
            const int tile_n0 = (tile % p.num_n_tiles) * BN;
            const int n0 = tile_n0 + (npart && part > 0 ? part * width : 0);
            // First output channel of accumulator columns [32c, 32c+32).  A part of
            // a paired MMA's tile reads width/2 rows of each CTA's half of the
            // filter block: its first width/2 columns are channels from the first
            // half, the rest from the second.
            auto chan = [&](int c) -> int {
                if (PAIR && npart) {
                    const int hw = width / 2, r0 = part * hw;
                    return tile_n0 + (c * 32 < hw ? r0 + c * 32 : BN / 2 + r0 + (c * 32 - hw));
                }
                return n0 + c * 32;
            };
            const int b = T::NACC == 2 ? local & 1 : 0;
            const uint32_t acc_phase = T::NACC == 2 ? (uint32_t)(local >> 1) & 1u : (uint32_t)local & 1u;
            const int slice_key = 8 * n0 + (npart ? p.parts : 0);   // the channels and width the slice must hold
            if (!b_res && p.epilogue == 1 && slice_key != slice_n0) {   // before the accumulator wait, which hides the latency
                float sv[kChunks], bv[kChunks];
#pragma unroll
                for (int i = 0; i < kChunks; ++i) {
                    const int c = h + i * (kEpiWarps / 4);
                    // chunks past the item's width (a tile part's) are not needed
                    // and channels past C_out (the last channel tile's) are masked
                    const bool in = c * 32 < width && chan(c) + lane < p.C_out;
                    sv[i] = in ? __ldg(p.scale + chan(c) + lane) : 0.0f;
                    bv[i] = in ? __ldg(p.bias + chan(c) + lane) : 0.0f;
                }
                __syncwarp();   // every lane is done with the previous tile's values
#pragma unroll
                for (int i = 0; i < kChunks; ++i) {
                    slice[i * 64 + lane] = sv[i];
                    slice[i * 64 + 32 + lane] = bv[i];
                }
                __syncwarp();
                slice_n0 = slice_key;
            }
            const bool got = ptx::mbar_wait(&tfull[b], acc_phase, p.wait_ns);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
#pragma unroll 1
            for (int hh = 0; hh < mh; ++hh) {
                const int prow = m0 + hh * BM + q * 32;   // first pixel of this warp's rows
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * MH * BN + hh * BN);
#pragma unroll 1
                for (int c = h, ci = 0; c * 32 < width; c += kEpiWarps / 4, ++ci) {
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(taddr + (uint32_t)(c * 32), r);
                    if (p.epilogue == 2) {
                        // split-K partial: this lane's row, 32 fp32 channels, 128 contiguous bytes
                        ptx::tmem_ld_wait();
                        const int m = prow + lane;
                        if (m < p.M) {
                            float4 *dst = reinterpret_cast<float4 *>(p.ws + ((int64_t)split * p.M + m) * p.C_out + chan(c));
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                     __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                        }
                        continue;
                    }
                    // the store issued from this box for the previous chunk must have read it
                    if (lane == 0) ptx::bulk_wait_group_read<0>();
                    __syncwarp();
                    ptx::tmem_ld_wait();
                    const int ch0 = chan(c);
                    const float4 *s4 = reinterpret_cast<const float4 *>(b_res ? table + (ch0 - cta_n0) : slice + ci * 64);
                    const float4 *b4 =
                        reinterpret_cast<const float4 *>(b_res ? table + BN + (ch0 - cta_n0) : slice + ci * 64 + 32);
                    uint32_t wq[4];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        float2 v0 = make_float2(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]));
                        float2 v1 = make_float2(__uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                        if (p.epilogue) {
                            const float4 a4 = s4[j], c4 = b4[j];
                            v0 = silu_f32x2(ffma2(v0, make_float2(a4.x, a4.y), make_float2(c4.x, c4.y)));
                            v1 = silu_f32x2(ffma2(v1, make_float2(a4.z, a4.w), make_float2(c4.z, c4.w)));
                        }
                        __nv_bfloat162 t0 = __floats2bfloat162_rn(v0.x, v0.y), t1 = __floats2bfloat162_rn(v1.x, v1.y);
                        wq[2 * (j & 1)] = *reinterpret_cast<uint32_t *>(&t0);
                        wq[2 * (j & 1) + 1] = *reinterpret_cast<uint32_t *>(&t1);
                        if (j & 1) {
                            // row `lane`, 16-byte chunk j/2 lands at chunk (j/2) ^ ((lane >> 1) & 3):
                            // the 64-byte swizzle the store's tensor map expects
                            const int pj = (j >> 1) ^ ((lane >> 1) & 3);
                            *reinterpret_cast<uint4 *>(box + lane * 64 + pj * 16) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
                        }
                    }
                    if (p.y_direct) {
                        // rows of y not 16-byte multiples: lane l copies channel ch0 + l of
                        // each of the box's 32 rows (64 contiguous bytes per row and store)
                        __syncwarp();
                        const bool col_ok = ch0 + lane < p.C_out;
                        uint16_t *y16 = reinterpret_cast<uint16_t *>(p.y);
#pragma unroll 4
                        for (int r = 0; r < 32; ++r) {
                            const int pj = (lane >> 3) ^ ((r >> 1) & 3);
                            const uint16_t v = *reinterpret_cast<const uint16_t *>(box + r * 64 + pj * 16 + (lane & 7) * 2);
                            if (col_ok && prow + r < p.M) y16[(int64_t)(prow + r) * p.C_out + ch0 + lane] = v;
                        }
                        __syncwarp();   // the box is read before the next chunk overwrites it
                    } else {
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            // the store clips at the tensor's edges (rows past M, channels
                            // past C_out); a box wholly past either is not issued
                            if (prow < p.M && ch0 < p.C_out) ptx::tma_store_2d(&tmap_y, box, ch0, prow);
                            ptx::bulk_commit_group();
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            if constexpr (PAIR) {
                __syncwarp();   // every lane's TMEM reads of this accumulator are done
                if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(&tempty[b], 0));
            } else {
                ptx::mbar_arrive(&tempty[b]);
            }
        }
        if (lane == 0) ptx::bulk_wait_group_all();   // stores complete before exit
        if (!ok && lane == 0) atomicOr(p.err, TF_DEVERR_EPILOGUE_WAIT);
    }

    ptx::tc_fence_before();
    cta_sync();
    // neither CTA of a pair frees its TMEM or exits while the pair's MMAs,
    // commits, copies or arrivals may still reach it
    if constexpr (PAIR) ptx::cluster_sync();
    if (warp == 1) {
        ptx::tc_fence_after();
        if constexpr (PAIR)
            ptx::tmem_dealloc_pair(tmem_base, T::TMEM_COLS);
        else
            ptx::tmem_dealloc(tmem_base, T::TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
using EncodeIm2colFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                    const cuuint64_t *, const int *, const int *, cuuint32_t, cuuint32_t,
                                    const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

template <typename Fn>
Fn driver_fn(const char *name)
{
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(fn);
}

EncodeTiledFn encode_tiled()
{
    static EncodeTiledFn fn = driver_fn<EncodeTiledFn>("cuTensorMapEncodeTiled");
    return fn;
}

EncodeIm2colFn encode_im2col()
{
    static EncodeIm2colFn fn = driver_fn<EncodeIm2colFn>("cuTensorMapEncodeIm2col");
    return fn;
}

// Channel tile width: the widest of 256/128/64/32 dividing C_out; for other
// channel counts the smallest of them covering C_out (256 beyond), so that
// only the last tile is partial.
int pick_bn(int C_out)
{
    if (C_out % 256 == 0) return 256;
    if (C_out % 128 == 0) return 128;
    if (C_out % 64 == 0) return 64;
    if (C_out % 32 == 0) return 32;
    for (int bn : {32, 64, 128})
        if (C_out <= bn) return bn;
    return 256;
}

bool is_plain_gemm(const tf_conv_shape &s)
{
    return s.KH == 1 && s.KW == 1 && s.stride_h == 1 && s.stride_w == 1 && s.pad_h == 0 && s.pad_w == 0;
}

// Upper corner of the im2col bounding box relative to the far edge, chosen so
// that the box, traversed with the conv stride, holds exactly Wo (Ho) base
// positions ow*stride - pad.
int upper_corner(int in, int out, int stride, int pad) { return (out - 1) * stride - pad - (in - 1); }

// Shared-memory plan for BN x EPI: the resident filter block when asked for
// and within kBResMaxBytes with at least 3 A stages left, else the plain
// ring; as many stages as fit, up to kMaxStages.  False if fewer than two fit.
template <int BN, int EPI, int MH = 1, int CG = 1>
bool plan_smem(int num_kb, bool want_bres, SmemPlan &sm)
{
    constexpr int kBoxes = EPI * kOutBoxBytes;
    constexpr int kSlices = EPI * chunks_per_warp(BN, EPI) * kParamChunkBytes;   // per-warp parameter slices
    constexpr int kTable = 2 * BN * 4;                                              // or one table (resident block)
    constexpr int b_bytes = Tile<BN, MH, CG>::B_BYTES;
    const int64_t bres_bytes = (int64_t)num_kb * b_bytes;
    sm.b_res = MH == 1 && want_bres && bres_bytes <= kBResMaxBytes &&
               (kSmemLimit - (kBoxes + kTable + kBarBytes) - bres_bytes) / kABytes >= 3;
    const int fixed = kBoxes + (sm.b_res ? kTable : kSlices) + kBarBytes;
    sm.stage_bytes = MH * kABytes + (sm.b_res ? 0 : b_bytes);
    const int64_t room = kSmemLimit - fixed - (sm.b_res ? bres_bytes : 0);
    sm.stages = (int)(room / sm.stage_bytes);
    const int cap = sm.b_res ? kMaxStages : kMaxStagesStreamed;
    if (sm.stages > cap) sm.stages = cap;
    if (sm.stages < 2) return false;
    sm.off_bres = sm.stages * sm.stage_bytes;
    sm.off_out = sm.off_bres + (sm.b_res ? (int)bres_bytes : 0);
    sm.off_par = sm.off_out + kBoxes;
    sm.off_bar = sm.off_par + (sm.b_res ? kTable : kSlices);
    sm.alloc = sm.off_bar + kBarBytes;
    return sm.alloc <= kSmemLimit;
}

// The last, partial wave of wide tiles as their 128-row halves over twice the
// units (CTAs, or CTA pairs), when that still fits in one wave (used when
// leave_wide_tail leaves nothing to a second launch).
inline void split_wide_tail(UmmaParams &p, int units)
{
    const int rem = p.num_tiles % units;
    if (rem > 0 && 2 * rem <= units) {
        p.split_from = p.num_tiles - rem;
        p.parts = 2;
        p.num_work = p.split_from + 2 * rem;
    }
}

// The last, partial wave of wide tiles, when it fills at most half the units,
// left to a second launch on 128-row tiles: on its own ring plan (one MMA per
// K step, more stages) such a tile keeps the tensor pipe fed, where the wide
// kernel's 128-row halves (48 KB stages carrying one MMA each) starve it.  The
// launch keeps whole 256-row blocks of tiles (all their channel tiles); false
// (and no change) when there is no such tail or no block would be left.
template <int CL, int MH>
bool leave_wide_tail(UmmaParams &p, int units, int *tail_row)
{
    if (!tail_row) return false;
    const int rem = p.num_tiles % units;
    if (rem == 0 || 2 * rem > units) return false;
    const int blocks = (p.num_tiles - rem) / p.num_n_tiles;   // 256-row blocks (per CTA) kept here
    if (blocks < 1) return false;
    p.num_tiles = blocks * p.num_n_tiles;
    p.num_work = p.num_tiles;
    p.split_from = p.num_work;
    p.parts = 1;
    *tail_row = p.m_base + blocks * CL * BM * MH;
    return true;
}

// The last, partial wave of tiles with a resident filter block and one
// channel tile as quarter or half tiles over 4 or 2 times the units, when that
// still fits in one wave; each part is at least `min_width` channels wide
// (measured 2-2.5% off the 1x1 workload's time on single CTAs).
inline void split_channel_tail(UmmaParams &p, int units, int bn, int min_width)
{
    const int rem = p.num_tiles % units;
    for (int parts : {4, 2}) {
        if (rem > 0 && parts * rem <= units && bn / parts >= min_width) {
            p.split_from = p.num_tiles - rem;
            p.parts = parts;
            p.num_work = p.split_from + parts * rem;
            return;
        }
    }
}

// With MH = 2 and tail_row given, a last partial wave of at most half the
// units is left out of this launch (whole 256-row blocks of tiles) and
// *tail_row set to its first output row, for the caller to run on 128-row
// tiles in a second launch; *tail_row stays 0 when this launch covers all.
template <int BN, bool IM2COL, int CL, int EPI, int MH = 1, int CG = 1>
cudaError_t launch_bn(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &ty, UmmaParams p,
                      bool want_bres, cudaStream_t st, int *tail_row = nullptr)
{
    constexpr int kThreads = threads_for(EPI);
    auto kern = conv_umma_kernel<BN, IM2COL, CL, EPI, MH, CG>;
    if (CG == 2 && p.splits != 1) return cudaErrorNotSupported;   // paired MMAs: one K split
    if constexpr (MH > 1) {   // 256-row tiles: one K split, no channel parts
        if (p.splits != 1) return cudaErrorNotSupported;
        const int64_t mtiles = ((int64_t)p.M + BM * MH - 1) / (BM * MH);
        p.num_tiles = (int)((mtiles + CL - 1) / CL) * p.num_n_tiles;
        p.num_work = p.num_tiles;
        p.split_from = p.num_work;
        p.parts = 1;
    }
    // the channel tiles cover C_out, and only the last one may be partial
    // (its filter rows past C_out zero-filled, its parameters masked, its
    // stores clipped): no filter box or store starts past the last channel
    if (p.num_n_tiles * BN < p.C_out || (p.num_n_tiles - 1) * BN >= p.C_out) return cudaErrorNotSupported;
    // a paired MMA's second CTA loads filter rows from BN/2 on: whole tiles only
    if (CG == 2 && p.num_n_tiles * BN != p.C_out) return cudaErrorNotSupported;
    if (!plan_smem<BN, EPI, MH, CG>(p.num_kb, want_bres && p.splits == 1, p.sm))
        return cudaErrorNotSupported;
    // Per-function, per-device attribute; cheap enough to set on every launch.
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, p.sm.alloc);
    if (e != cudaSuccess) return e;
    // programmatic dependent launch: the kernel's set-up may overlap the
    // previous kernel of the stream (it waits before touching global memory)
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = p.sm.alloc;
    cfg.stream = st;
    cfg.attrs = attr;
    if constexpr (CL == 1) {
        int grid = sm_count();
        // a resident filter block pins each CTA to one channel tile: launch a
        // multiple of num_n_tiles CTAs so that work c, c + grid, ... keeps
        // channel tile c % num_n_tiles
        if (p.sm.b_res) grid = grid / p.num_n_tiles * p.num_n_tiles;
        if (grid < 1) return cudaErrorNotSupported;
        if (MH > 1 && !leave_wide_tail<CL, MH>(p, grid, tail_row)) split_wide_tail(p, grid);
        if (MH == 1 && p.sm.b_res && p.num_n_tiles == 1 && p.C_out == BN && p.splits == 1)
            split_channel_tail(p, grid, BN, 32);
        if (grid > p.num_work) grid = p.num_work;
        cfg.gridDim = dim3((unsigned)grid);
        cfg.numAttrs = 1;
        return counted(cudaLaunchKernelEx(&cfg, kern, ta, tb, ty, p));
    } else {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = CL;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
        // persistent: as many clusters as can be resident at once (an SM left
        // without a partner in its GPC stays idle rather than starting a
        // second wave)
        cfg.gridDim = dim3(sm_count() / CL * CL);
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
        if (e != cudaSuccess) return e;
        // a resident filter block pins each pair to one channel tile
        if (p.sm.b_res) clusters = clusters / p.num_n_tiles * p.num_n_tiles;
        if (clusters < 1) return cudaErrorNotSupported;
        if (MH > 1 && !leave_wide_tail<CL, MH>(p, clusters, tail_row)) split_wide_tail(p, clusters);
        // a part of a paired MMA takes half its channels from each CTA's half
        // of the block, in whole 32-channel chunks: parts of >= 64 channels
        if (MH == 1 && p.sm.b_res && p.num_n_tiles == 1 && p.C_out == BN && p.splits == 1)
            split_channel_tail(p, clusters, BN, 64);
        if (clusters > p.num_work) clusters = p.num_work;
        cfg.gridDim = dim3(CL * clusters);
        return counted(cudaLaunchKernelEx(&cfg, kern, ta, tb, ty, p));
    }
}

template <bool IM2COL, int CL, int EPI, int CG = 1>
cudaError_t launch_epi(int bn, const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &ty,
                       const UmmaParams &p, bool want_bres, cudaStream_t st)
{
    switch (bn) {
    case 256: return launch_bn<256, IM2COL, CL, EPI, 1, CG>(ta, tb, ty, p, want_bres, st);
    case 128: return launch_bn<128, IM2COL, CL, EPI, 1, CG>(ta, tb, ty, p, want_bres, st);
    case 64: return launch_bn<64, IM2COL, CL, EPI, 1, CG>(ta, tb, ty, p, want_bres, st);
    case 32: return launch_bn<32, IM2COL, CL, EPI, 1, CG>(ta, tb, ty, p, want_bres, st);
    default: return cudaErrorNotSupported;
    }
}

// A work item of at most 16 K blocks finishes its MMAs in about the time the
// epilogue needs for the previous tile: such kernels get more epilogue warps.
bool short_k(int kb_per_split) { return kb_per_split <= 16; }

template <bool IM2COL, int CL, int CG = 1>
cudaError_t launch_im(int bn, const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &ty,
                      const UmmaParams &p, bool want_bres, cudaStream_t st)
{
    if (short_k(p.kb_per_split))
        return launch_epi<IM2COL, CL, kEpiWarpsShortK, CG>(bn, ta, tb, ty, p, want_bres, st);
    return launch_epi<IM2COL, CL, kEpiWarpsLongK, CG>(bn, ta, tb, ty, p, want_bres, st);
}

// Channel tile width: the widest of 256/128/64/32 dividing C_out, except that
// a short-K kernel (sixteen epilogue warps) on single CTAs takes 128 instead
// of 256 unless its whole filter block can stay resident: at 256 only three
// ring stages would fit beside the staging boxes.  (A paired MMA holds half
// the filter tile per CTA, so 256 leaves room for five.)
int choose_bn(const tf_conv_shape &s, int splits, int cl, bool pair_mma)
{
    int bn = pick_bn(s.C_out);
    const int num_kb = s.KH * s.KW * ((s.C_in + BK - 1) / BK);
    const int kb_per_split = (num_kb + splits - 1) / splits;
    if (bn == 256 && short_k(kb_per_split) && !pair_mma) {
        const bool resident = cl == 1 && splits == 1 && (int64_t)num_kb * Tile<256>::B_BYTES <= kBResMaxBytes;
        if (!resident) bn = 128;
    }
    return bn;
}

}  // namespace

bool conv_umma_supports(const tf_conv_shape &s, int Ho, int Wo)
{
    // any C_in the API takes (a multiple of 8: 16-byte rows for TMA); the last
    // 64-channel block of each filter tap is zero-filled past C_in
    if (s.C_in % 8 != 0 || s.C_out < 1) return false;
    if ((int64_t)s.N * Ho * Wo >= (int64_t)1 << 31) return false;
    if (is_plain_gemm(s)) return true;
    // im2col geometry: traversal strides up to 8, filter taps addressed by
    // 16-bit offsets, and bounding-box corners within the signed 8-bit range a
    // 4-D im2col tensor map takes.
    if (s.stride_h > 8 || s.stride_w > 8 || s.KH > 65535 || s.KW > 65535) return false;
    const int lw = -s.pad_w, uw = upper_corner(s.W, Wo, s.stride_w, s.pad_w);
    const int lh = -s.pad_h, uh = upper_corner(s.H, Ho, s.stride_h, s.pad_h);
    for (int c : {lw, uw, lh, uh})
        if (c < -128 || c > 127) return false;
    return true;
}

cudaError_t launch_conv_umma(const ConvArgs &a, cudaStream_t st)
{
    const tf_conv_shape &s = a.s;
    if (!conv_umma_supports(s, a.Ho, a.Wo)) return cudaErrorNotSupported;
    EncodeTiledFn tiled = encode_tiled();
    if (!tiled) return cudaErrorNotSupported;
    // a 2-CTA cluster always runs the paired MMA (each CTA holds half of B)
    const int cl = a.cluster == 2 ? 2 : 1;
    const bool pair = cl == 2;
    // wide (256-row) tiles: 256-channel tiles whatever the K length (the
    // kernel is built for BN = 256), no K split
    if (a.wide && (pick_bn(s.C_out) != 256 || a.splits > 1)) return cudaErrorNotSupported;
    if (pair && a.splits > 1) return cudaErrorNotSupported;
    // channel tails (C_out % 32 != 0) run on single CTAs without a K split
    if (s.C_out % 32 != 0 && (pair || a.splits > 1)) return cudaErrorNotSupported;
    const int bn = a.wide ? 256 : choose_bn(s, a.splits > 1 ? a.splits : 1, cl, pair);
    const int64_t M = (int64_t)s.N * a.Ho * a.Wo;
    const int taps = s.KH * s.KW;
    const int cblocks = (s.C_in + BK - 1) / BK;   // 64-channel K steps per filter tap
    const bool y_direct = s.C_out % 8 != 0;       // y rows not 16-byte multiples: no TMA store

    CUtensorMap ta, tb, ty;
    memset(&ty, 0, sizeof ty);
    if (!y_direct) {   // y: the NHWC output as a [M][C_out] matrix, stored in 32 x 32 boxes
        const cuuint64_t dims[2] = {(cuuint64_t)s.C_out, (cuuint64_t)M};
        const cuuint64_t strides[1] = {(cuuint64_t)s.C_out * 2};
        const cuuint32_t box[2] = {kOutBox, kOutBox};
        const cuuint32_t estr[2] = {1, 1};
        if (tiled(&ty, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.y, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {   // B: packed filters [C_out][tap][C_in] (OHWI); a box is 64 input channels of one
        // tap for BN output channels (half of them per CTA of a pair), K-major,
        // zero-filled past C_in and past C_out
        const cuuint64_t dims[3] = {(cuuint64_t)s.C_in, (cuuint64_t)taps, (cuuint64_t)s.C_out};
        const cuuint64_t strides[2] = {(cuuint64_t)s.C_in * 2, (cuuint64_t)taps * s.C_in * 2};
        const cuuint32_t box[3] = {BK, 1, (cuuint32_t)(pair ? bn / 2 : bn)};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (tiled(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.w), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const bool im2col = !is_plain_gemm(s);
    if (!im2col) {   // A: the input itself is the [M][C_in] matrix
        const cuuint64_t dims[2] = {(cuuint64_t)s.C_in, (cuuint64_t)M};
        const cuuint64_t strides[1] = {(cuuint64_t)s.C_in * 2};
        const cuuint32_t box[2] = {BK, BM};
        const cuuint32_t estr[2] = {1, 1};
        if (tiled(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(a.x), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    } else {         // A: im2col view of the NHWC input
        EncodeIm2colFn enc = encode_im2col();
        if (!enc) return cudaErrorNotSupported;
        const cuuint64_t dims[4] = {(cuuint64_t)s.C_in, (cuuint64_t)s.W, (cuuint64_t)s.H, (cuuint64_t)s.N};
        const cuuint64_t strides[3] = {(cuuint64_t)s.C_in * 2, (cuuint64_t)s.W * s.C_in * 2,
                                       (cuuint64_t)s.H * s.W * s.C_in * 2};
        const int lower[2] = {-s.pad_w, -s.pad_h};
        const int upper[2] = {upper_corner(s.W, a.Wo, s.stride_w, s.pad_w), upper_corner(s.H, a.Ho, s.stride_h, s.pad_h)};
        const cuuint32_t estr[4] = {1, (cuuint32_t)s.stride_w, (cuuint32_t)s.stride_h, 1};
        if (enc(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(a.x), dims, strides, lower, upper, BK,
                BM, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }

    UmmaParams p;
    p.scale = a.scale;
    p.bias = a.bias;
    p.y = reinterpret_cast<__nv_bfloat16 *>(a.y);
    p.err = device_error_word();
    p.wait_ns = wait_limit_ns();
    p.M = (int)M;
    p.m_base = 0;
    p.C_out = s.C_out;
    p.KW = s.KW;
    p.HoWo = a.Ho * a.Wo;
    p.Wo = a.Wo;
    p.stride_h = s.stride_h;
    p.stride_w = s.stride_w;
    p.pad_h = s.pad_h;
    p.pad_w = s.pad_w;
    p.cblocks = cblocks;
    p.num_kb = taps * cblocks;
    p.num_n_tiles = (s.C_out + bn - 1) / bn;
    p.num_tiles = (int)(((M + BM - 1) / BM + cl - 1) / cl) * p.num_n_tiles;   // cl vertically adjacent tiles each
    p.epilogue = a.epilogue;
    p.y_direct = y_direct ? 1 : 0;
    p.splits = 1;
    p.kb_per_split = p.num_kb;
    p.ws = nullptr;
    if (a.splits > 1) {
        if (!a.ws) return cudaErrorInvalidValue;
        p.kb_per_split = (p.num_kb + a.splits - 1) / a.splits;
        p.splits = (p.num_kb + p.kb_per_split - 1) / p.kb_per_split;   // no empty split
        p.epilogue = 2;
        p.ws = a.ws;
    }
    p.num_work = p.num_tiles * p.splits;
    p.split_from = p.num_work;   // no tile parts unless launch_bn decides so
    p.parts = 1;
    if (p.err == nullptr) return cudaErrorInitializationError;
    const bool want_bres = p.splits == 1;
    if (a.wide) {
        // the wide kernel, then (when it leaves one) its partial last wave on
        // 128-row tiles of the same CTA grouping
        int tail_row = 0;
        cudaError_t e;
        if (pair)
            e = im2col ? launch_bn<256, true, 2, kEpiWarpsLongK, 2, 2>(ta, tb, ty, p, false, st, &tail_row)
                       : launch_bn<256, false, 2, kEpiWarpsLongK, 2, 2>(ta, tb, ty, p, false, st, &tail_row);
        else
            e = im2col ? launch_bn<256, true, 1, kEpiWarpsLongK, 2>(ta, tb, ty, p, false, st, &tail_row)
                       : launch_bn<256, false, 1, kEpiWarpsLongK, 2>(ta, tb, ty, p, false, st, &tail_row);
        if (e != cudaSuccess || tail_row == 0) return e;
        UmmaParams t = p;
        t.m_base = tail_row;
        t.num_tiles = (int)((((int64_t)M - tail_row + BM - 1) / BM + cl - 1) / cl) * t.num_n_tiles;
        t.num_work = t.num_tiles;
        t.split_from = t.num_work;
        t.parts = 1;
        if (pair)
            return im2col ? launch_bn<256, true, 2, kEpiWarpsLongK, 1, 2>(ta, tb, ty, t, false, st)
                          : launch_bn<256, false, 2, kEpiWarpsLongK, 1, 2>(ta, tb, ty, t, false, st);
        return im2col ? launch_bn<256, true, 1, kEpiWarpsLongK, 1>(ta, tb, ty, t, false, st)
                      : launch_bn<256, false, 1, kEpiWarpsLongK, 1>(ta, tb, ty, t, false, st);
    }
    if (pair)
        return im2col ? launch_im<true, 2, 2>(bn, ta, tb, ty, p, want_bres, st)
                      : launch_im<false, 2, 2>(bn, ta, tb, ty, p, want_bres, st);
    return im2col ? launch_im<true, 1>(bn, ta, tb, ty, p, want_bres, st)
                  : launch_im<false, 1>(bn, ta, tb, ty, p, want_bres, st);
}

// ---------------------------------------------------------------- split K

int conv_umma_splits(const tf_conv_shape &s, int Ho, int Wo)
{
    // whole channel tiles only: the fp32 partials are written as 128-byte rows
    if (s.C_out % 32 != 0) return 1;
    const int bn = pick_bn(s.C_out);
    const int64_t M = (int64_t)s.N * Ho * Wo;
    const int64_t tiles = (M + BM - 1) / BM * (s.C_out / bn);
    const int64_t num_kb = (int64_t)s.KH * s.KW * ((s.C_in + BK - 1) / BK);
    const int sms = sm_count();
    if (tiles * 2 > sms) return 1;          // at least half the SMs busy already
    if (num_kb < 16) return 1;              // short K loops: the extra reduction costs more than it saves
    int64_t S = sms / tiles;
    if (S > num_kb / 4) S = num_kb / 4;     // at least 4 K blocks per split
    if (S < 2) return 1;
    const int64_t kbps = (num_kb + S - 1) / S;
    return (int)((num_kb + kbps - 1) / kbps);
}

namespace {
// y = epilogue(sum over splits of the fp32 partials), 8 channels per thread.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float *__restrict__ ws, int splits, int64_t MC,
                                                            int C_out, const float *__restrict__ scale,
                                                            const float *__restrict__ bias,
                                                            __nv_bfloat16 *__restrict__ y, int epilogue)
{
    pdl_begin();
    const int64_t nvec = MC / 8;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
        float v[8];
        const float4 *src = reinterpret_cast<const float4 *>(ws) + 2 * i;
        float4 a = __ldcs(src), b = __ldcs(src + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        for (int sidx = 1; sidx < splits; ++sidx) {
            const float4 *q = reinterpret_cast<const float4 *>(ws + sidx * MC) + 2 * i;
            a = __ldcs(q);
            b = __ldcs(q + 1);
            v[0] += a.x; v[1] += a.y; v[2] += a.z; v[3] += a.w; v[4] += b.x; v[5] += b.y; v[6] += b.z; v[7] += b.w;
        }
        const int c0 = (int)((8 * i) % C_out);
        uint4 o;
        __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&o);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float2 t = make_float2(v[2 * j], v[2 * j + 1]);
            if (epilogue)
                t = silu_f32x2(ffma2(t, make_float2(__ldg(scale + c0 + 2 * j), __ldg(scale + c0 + 2 * j + 1)),
                                     make_float2(__ldg(bias + c0 + 2 * j), __ldg(bias + c0 + 2 * j + 1))));
            h[j] = __floats2bfloat162_rn(t.x, t.y);
        }
        reinterpret_cast<uint4 *>(y)[i] = o;
    }
}
}  // namespace

cudaError_t launch_splitk_reduce(const float *ws, int splits, int64_t M, int C_out, const float *scale,
                                 const float *bias, void *y, int epilogue, cudaStream_t st)
{
    const int64_t MC = M * C_out;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, splitk_reduce_kernel, 256, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    int64_t grid = (MC / 8 + 255) / 256;
    if (grid > (int64_t)sm_count() * per_sm) grid = (int64_t)sm_count() * per_sm;
    return launch_pdl(splitk_reduce_kernel, dim3((unsigned)grid), dim3(256), 0, st, ws, splits, MC, C_out, scale, bias,
                      reinterpret_cast<__nv_bfloat16 *>(y), epilogue);
}

// ---------------------------------------------------------------- wait probe

namespace {
__global__ void wait_probe_kernel(uint32_t *err, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        ptx::mbar_init_fence();
    }
    cta_sync();
    // Nothing ever arrives on `bar`: phase 0 never completes, the wait gives up.
    if (threadIdx.x == 0 && !ptx::mbar_wait(&bar, 0, limit_ns)) atomicOr(err, TF_DEVERR_PROBE_WAIT);
}
}  // namespace

cudaError_t launch_wait_probe(uint64_t limit_ns, cudaStream_t st)
{
    uint32_t *err = device_error_word();
    if (err == nullptr) return cudaErrorInitializationError;
    wait_probe_kernel<<<1, 32, 0, st>>>(err, limit_ns);
    return counted(cudaGetLastError());
}

}  // namespace tf
