// gemv_m1.cu -- Q4_K decode GEMV for one activation row (y = W x), the
// kernel that streams the weights of a batch-1 decode step.
//
// The operation: "Building a Rust Inference Engine That Matches Llama.cpp",
// "Where the wins came from" -- the dequantisation is paid once, inside the
// dot product, never as a separate memory-bound pass over a decoded buffer.
//
// Arithmetic (the one-row operand form of tc_common.cuh, unit_dot_sb): the
// nibbles enter mma.sync.m16n8k16 unscaled, as fp16 subnormals (w & 0x000F000F
// is the half pair (q0, q1) * 2^-24, w & 0x00F000F0 is (q0, q1) * 2^-20), and
// the activations as two fp16 terms (hi + lo) after an exact power-of-two
// scale per super-block, so every product is exact and only the fp32
// accumulation rounds.  Lane column c of an MMA carries sub-block 2c (low
// nibbles) or 2c+1 (high nibbles); B column pair (2c, 2c+1) holds the hi and
// lo terms of that sub-block's activations, zeros elsewhere.  Each lane then
// applies d*sc and dmin*m once per (row, sub-block) in fp32, for its two rows
// g and g+8 together in packed fp32 (FFMA2):
//   y_r += d * 2^-s * (sc_2c * 2^24 * D_lo + sc_2c+1 * 2^20 * D_hi)
//          - dmin * (m_2c * X_2c + m_2c+1 * X_2c+1)
// with X_j the fp32 sum of sub-block j's activations.
//
// Work decomposition.  The 16-row tiles of all matrices of a group (they
// share x) are concatenated (T tiles); K may be cut into S slices of KS
// super-blocks (only when x's layout for the whole K would crowd the ring
// out of shared memory).  A work item is TS consecutive tiles x one slice,
// taken in NP passes of WS super-blocks; one pass is WS*TS units of 16 rows x
// 256 weights (2304 bytes each), exactly one ring slot.  CTA b works on slice
// b % S.  Items are handed out in two phases: each CTA's
// first F items are fixed (so that its producer can fetch them before the
// previous kernel in the stream has finished), the rest come from a counter
// per slice, so CTAs on faster SMs take more.  Each item is computed whole by
// one CTA, in a fixed order: results do not depend on the schedule.
//
// Inside a CTA one producer warp and W = WS*TS consumer warps:
//  - the producer fills a ring of slots with one TMA box per tile, through
//    a 3-D view of the matrix (144-byte super-block, row, super-block index)
//    that lands the tile as WS units of 16 rows x 144 bytes -- rows 144 bytes
//    apart, so the lanes reading the same column of neighbouring rows hit
//    different banks -- completing on the slot's mbarrier.  It writes the
//    slot's item index and pass first, and a negative index once the work has
//    run out;
//  - consumer warp w always takes unit w = (tile w / WS, super-block w % WS
//    of the pass) of a slot; with one pass its B fragments stay in registers
//    for the whole launch, with several it reloads them from shared memory
//    for each pass.  It copies its unit to registers, releases the slot, runs
//    16 MMAs and the scaling, and adds the two rows it covers into the column
//    of partial sums of its super-block position (passes in order);
//  - at the end the columns are added in column order and, with S > 1, the
//    slices in slice order by the CTA that finished an item's last slice (a
//    ticket per item): no float atomics, bitwise repeatable.
// The last CTA of a slice to stop fetching resets its counters, and counters
// are touched only after the previous kernel has completed, so back-to-back
// launches and CUDA-graph replays each start from zero.
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include <cuda.h>

#include "formats.cuh"
#include "qmm_device.cuh"
#include "qmm_internal.h"
#include "m1_device.cuh"
#include "tc_common.cuh"

namespace qmm {

namespace {

using namespace tc;
using namespace m1;

constexpr int kM1MaxSlots = kMaxSlots;
constexpr int kM1MaxShare = 16;  // average items per CTA at most

struct M1Params {
    CUtensorMap tmap[kMaxGroup];  // 3-D column view of each matrix, box (18, 16, WS)
    int tile_end[kMaxGroup];      // cumulative 16-row tile counts
    int rows[kMaxGroup];
    float *y[kMaxGroup];
    const float *x;
    float *ws;                    // [S][T*16] K-slice partial sums (S > 1)
    unsigned *ctr;                // [S] next item, [S] CTAs done, [n_items] item tickets (S > 1)
    unsigned *status;
    int T, nmat;
    int S, KS;                    // K slices, super-blocks per slice
    int WS, NP;                   // super-blocks per pass, passes (KS = WS * NP)
    int TS, W;                    // tiles per item, consumer warps (WS * TS)
    int G1;                       // CTAs per slice
    int n_items;                  // items per slice (ceil(T / TS))
    int F;                        // fixed items per CTA
    int cap;                      // items a CTA may take
    int nslot, slot_bytes;
};

__device__ __forceinline__ float silu(float z) { return z / (1.f + expf(-z)); }

// FUSE: the (gate, up) pair with its tiles interleaved (gate tile t at 2t,
// up tile t at 2t+1).
template <bool FUSE>
__device__ __forceinline__ int mat_of_tile(const M1Params &P, int t)
{
    if (FUSE)
        return t & 1;
    int m = 0;
#pragma unroll
    for (int i = 0; i < kMaxGroup - 1; ++i)
        if (i < P.nmat - 1 && t >= P.tile_end[i])
            m = i + 1;
    return m;
}

// Global row (tile*16 + r) -> (matrix, row of the matrix); false if the tile
// is the ragged end of a matrix and the row does not exist.
template <bool FUSE>
__device__ __forceinline__ bool locate_row(const M1Params &P, int tile, int r, int &m, int &row)
{
    m = mat_of_tile<FUSE>(P, tile);
    row = (FUSE ? tile >> 1 : tile - (m == 0 ? 0 : P.tile_end[m - 1])) * kTileRows + r;
    return row < P.rows[m];
}

template <int FMT, int UPW>
__global__ void __launch_bounds__(32 * (kM1MaxWarps + 1)) gemv_m1_kernel(const __grid_constant__ M1Params P)
{
    // super-block bytes, one unit's bytes (16 rows), offset of the nibbles,
    // activation sums per super-block (Q6_K: one per 16-weight group)
    constexpr bool Q6 = FMT == QMM_Q6_K;
    constexpr bool IQ = FMT == QMM_IQ4_NL;
    constexpr bool Q8 = FMT == QMM_Q8_0;
    constexpr int SB = FMT == QMM_Q5_K ? 176 : (Q6 ? 210 : (Q8 ? 272 : 144));
    constexpr int UB = kTileRows * SB;
    constexpr int QOFF = FMT == QMM_Q5_K ? 48 : 16;
    constexpr int XN = Q6 ? 16 : 8;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = __shfl_sync(0xffffffffu, int(threadIdx.x >> 5), 0);  // warp-uniform
    const int lane = threadIdx.x & 31;
    const int W = P.W, NS = P.nslot, KS = P.KS, TS = P.TS, WS = P.WS, NP = P.NP;
    // UPW: units per consumer warp and slot (WS * TS = W * UPW); two only for
    // the fused (gate, up) pair: the gate unit and the up unit of the same
    // rows and super-block, y[0] receiving silu(gate) * up
    constexpr bool FUSE = UPW == 2;
    const int b1 = int(blockIdx.x) / P.S, sl = int(blockIdx.x) - b1 * P.S;
    const int sb0 = sl * KS;
    const int itile = TS * kTileRows;  // rows of one item

    // Shared memory: ring [NS][slot_bytes] | Bx [KS][8][4][2] uint4 | Xs [KS][XN]
    // | inv [KS] | part [WS][cap*TS*16] | items [cap] | flags [cap] | full[NS],
    // empty[NS]
    uint8_t *ring = smem;
    uint4 *Bx = reinterpret_cast<uint4 *>(smem + size_t(NS) * P.slot_bytes);
    float *Xs = reinterpret_cast<float *>(Bx + size_t(KS) * 64);
    float *inv = Xs + size_t(KS) * XN;
    float *part = inv + ((KS + 3) & ~3);
    const int pcol = P.cap * itile;  // floats per column of partial sums
    int *items = reinterpret_cast<int *>(part + size_t(WS) * pcol);
    int *flags = items + P.cap;
    uint64_t *full = reinterpret_cast<uint64_t *>(
        (reinterpret_cast<uintptr_t>(flags + P.cap) + 7) & ~uintptr_t(7));
    uint64_t *empty = full + NS;
    __shared__ int s_item[kM1MaxSlots];
    __shared__ int s_pass[kM1MaxSlots];
    __shared__ int s_abort;
    __shared__ int s_issued;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], unsigned(32 * W));  // every consumer lane arrives
        }
        fence_barrier_init();
        s_abort = 0;
        s_issued = 0;
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == W) {
        // ---------------------------------------------------------- producer
        const uint64_t pol = policy_evict_first();
        int k = 0, slot = 0;
        unsigned par = 0;
        bool ok = true;
        // One slot: pass p of item `it` (negative: no more work).
        auto issue = [&](int it, int p) {
            if (k >= NS && !mbar_wait_polled(&empty[slot], par ^ 1u)) {
                if (lane == 0) {
                    atomicOr(P.status, kStatusTimeoutBit);
                    *(volatile int *)&s_abort = 1;
                }
                ok = false;
                return;
            }
            if (lane == 0) {
                s_item[slot] = it;
                s_pass[slot] = p;
            }
            if (it >= 0) {
                // Lane u < TS copies tile it*TS + u: one box of 16 rows x the
                // pass's WS super-blocks, landing as units u*WS .. u*WS+WS-1
                // (rows past a matrix end read as zeros and count in full
                // towards the transaction bytes).
                const int tile = it * TS + lane;
                const bool mine = lane < TS && tile < P.T;
                const int nvalid = __popc(__ballot_sync(0xffffffffu, mine));
                if (lane == 0)
                    mbar_arrive_expect_tx(&full[slot], unsigned(nvalid * WS) * UB);
                __syncwarp();
                if (mine) {
                    const int m = mat_of_tile<FUSE>(P, tile);
                    const int lt = FUSE ? tile >> 1 : tile - (m == 0 ? 0 : P.tile_end[m - 1]);
                    if constexpr (Q6)  // 16 rows x 8 super-blocks (1680 bytes), row-major
                        tma_load_2d(ring + size_t(slot) * P.slot_bytes + size_t(lane) * WS * UB,
                                    &P.tmap[m], ((sb0 + p * WS) / 8) * 210, lt * kTileRows,
                                    &full[slot], pol);
                    else
                        tma_load_3d(ring + size_t(slot) * P.slot_bytes + size_t(lane) * WS * UB,
                                    &P.tmap[m], lt * kTileRows, sb0 + p * WS, &full[slot], pol);
                }
            } else if (lane == 0) {
                mbar_arrive(&full[slot]);  // completes the phase with no bytes
            }
            __syncwarp();
            ++k;
            if (++slot == NS) {
                slot = 0;
                par ^= 1u;
            }
        };
        unsigned *next = P.ctr + sl, *done = P.ctr + P.S + sl;
        // Fixed items f*G1 + b1 (f < nfix); then dynamic items from the
        // counter.  `reserved` (lane 0) counts the items this CTA will compute
        // -- its fixed ones plus every index fetched -- and never exceeds cap,
        // so no fetched index is left uncomputed.  Two fetches are kept in
        // flight so that the atomics' round trips overlap the copies
        // (INT_MAX: nothing fetched).
        // fixed item f of this CTA: f*G1 + b1 (interleaved, so that every CTA
        // has its share even when F*G1 overshoots the items)
        const int nfix = b1 < P.n_items ? min(P.F, (P.n_items - b1 + P.G1 - 1) / P.G1) : 0;
        const int dyn0 = P.G1 * P.F;
        int reserved = nfix;
        int n0 = 0x7fffffff, n1 = 0x7fffffff;
        auto fetch = [&]() {
            if (reserved >= P.cap)
                return 0x7fffffff;
            ++reserved;
            return dyn0 + int(atomicAdd(next, 1u));
        };
        bool waited = false;
        auto start_dynamic = [&]() {
            // Counters are shared with earlier launches: touch them only
            // after those have completed.
            pdl_wait();
            waited = true;
            if (lane == 0) {
                n0 = fetch();
                n1 = fetch();
            }
        };
        // The fixed items' first NS slots are fetched before the previous
        // kernel has finished.
        for (int f = 0; f < nfix && ok; ++f)
            for (int p = 0; p < NP && ok; ++p) {
                if (k == NS && !waited)
                    start_dynamic();
                issue(f * P.G1 + b1, p);
            }
        if (!waited)
            start_dynamic();
        while (ok && !*(volatile int *)&s_abort) {
            const int it = __shfl_sync(0xffffffffu, n0, 0);
            if (it >= P.n_items)
                break;  // later fetches of this CTA return larger indices
            if (lane == 0) {
                n0 = n1;
                n1 = fetch();
            }
            for (int p = 0; p < NP && ok; ++p)
                issue(it, p);
        }
        if (lane == 0 && atomicAdd(done, 1u) == unsigned(P.G1 - 1)) {
            *next = 0u;  // every CTA of this slice has stopped fetching
            *done = 0u;
        }
        if (ok)
            issue(-1, 0);
        if (lane == 0)
            s_issued = k;
    } else {
        // ---------------------------------------------------------- consumers
        pdl_wait();  // x, y and the workspace belong to earlier kernels until here
        {
            // This slice of x -> B entries; super-blocks j = warp, warp + W, ...,
            // the loads of up to four in flight together.
            const int cc = lane >> 3, tt = lane & 7;
            // v: the weights of chunk cc's low nibbles, w (xb + wo): of its
            // high nibbles
            // (IQ4_NL: k-step tt of lane column cc reads code bytes
            // 4(tt & 3) .. +3 of block 2cc + tt / 4: low-nibble weights there,
            // high-nibble ones 16 further)
            const float *xb = P.x + int64_t(sb0) * 256 +
                              (Q6   ? 128 * (cc >> 1) + 32 * (cc & 1) + 4 * tt
                               : IQ ? 64 * cc + 32 * (tt >> 2) + 4 * (tt & 3)
                                    : 64 * cc + 4 * tt);
            constexpr int wo = Q6 ? 64 : (IQ ? 16 : 32);
            for (int j0 = warp; j0 < KS; j0 += 4 * W) {
                float4 v[4], w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int j = j0 + i * W;
                    if (j < KS) {
                        v[i] = __ldg(reinterpret_cast<const float4 *>(xb + int64_t(j) * 256));
                        w[i] = __ldg(reinterpret_cast<const float4 *>(xb + int64_t(j) * 256 + wo));
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int j = j0 + i * W;
                    if (j < KS)
                        prep_sb<Q6 ? 1 : (IQ ? 2 : (Q8 ? 3 : 0))>(v[i], w[i], lane, Bx + size_t(j) * 64,
                                                        Xs + j * XN, inv + j);
                }
            }
        }
        named_sync(1, W * 32);

        const int g = lane >> 2, c = lane & 3;
        const int wsb = warp % WS, wt = warp / WS;
        const bool act = (g >> 1) == c;
        const int term = g & 1;
        const ScaleSel L = scale_sel(c);
        // IQ4_NL: the code book as u = book + 128 bytes
        const Iq4Book book = {fmt::iq4nl_book_word(0) ^ 0x80808080u,
                              fmt::iq4nl_book_word(4) ^ 0x80808080u,
                              fmt::iq4nl_book_word(8) ^ 0x80808080u,
                              fmt::iq4nl_book_word(12) ^ 0x80808080u};
        // B fragments, sub-block sums and inverse scale of this warp's
        // super-block of pass p (reloaded per pass when there are several).
        uint4 B[8];
        float2 X0, X1, iv;
        float4 X6;  // Q6_K: the sums of the lane column's four 16-weight groups
        const int g6 = 8 * (c >> 1) + 2 * (c & 1);
        auto load_b = [&](int p) {
            const int j = p * WS + wsb;
#pragma unroll
            for (int t = 0; t < 8; ++t)
                B[t] = act ? Bx[size_t(j) * 64 + (t * 4 + c) * 2 + term] : make_uint4(0u, 0u, 0u, 0u);
            if constexpr (Q6) {
                X6 = make_float4(Xs[j * XN + g6], Xs[j * XN + g6 + 1], Xs[j * XN + g6 + 4],
                                 Xs[j * XN + g6 + 5]);
            } else if constexpr (IQ || Q8) {
                X0 = make_float2(Xs[j * XN + 2 * c], Xs[j * XN + 2 * c + 1]);  // blocks 2c, 2c+1
            } else {
                X0 = make_float2(Xs[j * XN + 2 * c], Xs[j * XN + 2 * c]);
                X1 = make_float2(Xs[j * XN + 2 * c + 1], Xs[j * XN + 2 * c + 1]);
            }
            iv = make_float2(inv[j], inv[j]);
        };
        load_b(0);
        const int slot_bytes = P.slot_bytes;
        // This lane's bytes of its unit in slot 0: header of row g (and of
        // row g+8 at +8*SB), its 32-byte nibble chunk at +QOFF+32c (Q5_K: the
        // 32 fifth-bit bytes at +16).
        // Q6_K: a tile's box is 16 rows of WS (= 8) super-blocks, row-major.
        const uint32_t ubase =
            smem_u32(ring) + uint32_t(Q6 ? wt * WS * UB + g * WS * SB + wsb * SB : warp * UB + g * SB);
        // Column wsb of the partial sums; lanes c = 0 and 1 own rows g and
        // g+8 of tile wt of the item.
        const uint32_t pbase =
            smem_u32(part + size_t(wsb) * pcol + wt * kTileRows + g + 8 * (c & 1));
        const bool writer = c < 2;
        uint32_t soff = 0;  // byte offset of the current slot
        unsigned par = 0;
        int slot = 0, k = 0;  // k: items completed by this CTA
        for (;;) {
            if (!mbar_wait_bounded(&full[slot], par)) {
                if (lane == 0) {
                    atomicOr(P.status, kStatusTimeoutBit);
                    *(volatile int *)&s_abort = 1;
                }
                break;
            }
            const int it = *(volatile int *)&s_item[slot];
            if (it < 0)
                break;
            const int p = *(volatile int *)&s_pass[slot];
            int kc = 0;
            // Units w, w + W, ... of the slot (UPW of them; the same
            // super-block, tiles wt, wt + W/WS, ...), one after the other; the
            // slot is released once the last one is in registers.
#pragma unroll
            for (int u = 0; u < UPW; ++u) {
            const int tl = wt + u * (W / WS);  // tile of the item
            const uint32_t a0 = ubase + soff + uint32_t(u * W * UB);
            uint32_t q6a[8], q6ha[8], q6b[8], q6hb[8], s6a = 0, s6b = 0, d6 = 0;
            if constexpr (Q6) {
                const uint32_t a1 = a0 + 8 * WS * SB;  // row g + 8
                const int n = c >> 1, s2 = 2 * (c & 1);
                q6_load(a0, c, q6a, q6ha);
                q6_load(a1, c, q6b, q6hb);
                s6a = lds_u16(a0 + 192 + 8 * n + s2) | (lds_u16(a0 + 196 + 8 * n + s2) << 16);
                s6b = lds_u16(a1 + 192 + 8 * n + s2) | (lds_u16(a1 + 196 + 8 * n + s2) << 16);
                d6 = lds_u16(a0 + 208) | (lds_u16(a1 + 208) << 16);
            }
            // (Q4_K / Q5_K units are 16-byte aligned; Q6_K's were read above)
            uint32_t q8a[17], q8b[17];
            if constexpr (Q8) {
#pragma unroll
                for (int q = 0; q < 17; ++q) {
                    q8a[q] = lds32(a0 + 68 * c + 4 * q);
                    q8b[q] = lds32(a0 + 8 * SB + 68 * c + 4 * q);
                }
            }
            uint32_t iwa[9], iwb[9];
            if constexpr (IQ) {
#pragma unroll
                for (int q = 0; q < 9; ++q) {
                    iwa[q] = lds32(a0 + 36 * c + 4 * q);
                    iwb[q] = lds32(a0 + 8 * SB + 36 * c + 4 * q);
                }
            }
            uint4 h0, h1, qa0, qa1, qb0, qb1, ha0, ha1, hb0, hb1;
            if constexpr (!Q6 && !IQ && !Q8) {
                h0 = lds128(a0);
                h1 = lds128(a0 + 8 * SB);
                qa0 = lds128(a0 + QOFF + 32 * c);
                qa1 = lds128(a0 + QOFF + 16 + 32 * c);
                qb0 = lds128(a0 + 8 * SB + QOFF + 32 * c);
                qb1 = lds128(a0 + 8 * SB + QOFF + 16 + 32 * c);
            }
            if constexpr (FMT == QMM_Q5_K) {
                ha0 = lds128(a0 + 16);
                ha1 = lds128(a0 + 32);
                hb0 = lds128(a0 + 8 * SB + 16);
                hb1 = lds128(a0 + 8 * SB + 32);
            }
            if (u == UPW - 1) {
                mbar_arrive(&empty[slot]);  // the units are in registers: release the slot
                soff += uint32_t(slot_bytes);
                if (++slot == NS) {
                    slot = 0;
                    soff = 0;
                    par ^= 1u;
                }
            }
            if (u == 0) {
                if (NP > 1)
                    load_b(p);
                kc = k;
                if (p == NP - 1)
                    ++k;
                if (p == 0 && warp == 0 && lane == 0)
                    items[kc] = it;
            }
            if (it * TS + tl >= P.T)
                continue;  // past the last tile (a ragged final item)
            float keep;
            if constexpr (Q8)
                keep = unit_rows_q8(q8a, q8b, B, c, X0, iv);
            else if constexpr (IQ)
                keep = unit_rows_iq4(iwa, iwb, book, B, c, X0, iv);
            else if constexpr (Q6)
                keep = unit_rows6(q6a, q6ha, q6b, q6hb, s6a, s6b, d6, B, c, X6, iv);
            else if constexpr (FMT == QMM_Q5_K)
                keep = unit_rows5(h0, h1, qa0, qa1, qb0, qb1, ha0, ha1, hb0, hb1, B, L, c, X0, X1,
                                  iv);
            else
                keep = unit_rows(h0, h1, qa0, qa1, qb0, qb1, B, L, c, X0, X1, iv);
            const uint32_t pa = pbase + uint32_t((kc * itile + u * (W / WS) * kTileRows) * 4);
            if (p > 0)
                keep = lds_f32_if(pa, writer) + keep;  // passes added in order
            sts_f32_if(pa, keep, writer);
            }
        }
        named_sync(1, W * 32);

        // ---- output: add the columns in column order, then (S > 1) the slices
        const int nrow = k * itile;
        // fused: row i of a gate tile pairs with row i + 16 (its up tile)
        auto store = [&](int tile, int r, float sg, float su) {
            int m, row;
            if (locate_row<FUSE>(P, tile, r, m, row))
                P.y[m][row] = FUSE ? silu(sg) * su : sg;
        };
        if (P.S == 1) {
            for (int i = threadIdx.x; i < nrow; i += W * 32) {
                const int tile = items[i / itile] * TS + (i % itile) / kTileRows;
                if (tile >= P.T || (FUSE && (tile & 1)))
                    continue;
                float s = 0.f, su = 0.f;
                for (int w = 0; w < WS; ++w)
                    s += part[size_t(w) * pcol + i];
                if (FUSE)
                    for (int w = 0; w < WS; ++w)
                        su += part[size_t(w) * pcol + i + kTileRows];
                store(tile, i % kTileRows, s, su);
            }
        } else {
            const size_t sst = size_t(P.T) * kTileRows;
            unsigned *tick = P.ctr + 2 * P.S;
            for (int i = threadIdx.x; i < nrow; i += W * 32) {
                const int tile = items[i / itile] * TS + (i % itile) / kTileRows;
                if (tile >= P.T)
                    continue;
                float s = 0.f;
                for (int w = 0; w < WS; ++w)
                    s += part[size_t(w) * pcol + i];
                __stcg(P.ws + size_t(sl) * sst + size_t(tile) * kTileRows + i % kTileRows, s);
            }
            __threadfence();
            named_sync(1, W * 32);
            for (int i = threadIdx.x; i < k; i += W * 32)
                flags[i] = atomicAdd(&tick[items[i]], 1u) == unsigned(P.S - 1) ? 1 : 0;
            named_sync(1, W * 32);
            __threadfence();
            for (int i = threadIdx.x; i < nrow; i += W * 32) {
                if (!flags[i / itile])
                    continue;
                const int tile = items[i / itile] * TS + (i % itile) / kTileRows;
                if (tile >= P.T || (FUSE && (tile & 1)))
                    continue;
                float s = 0.f, su = 0.f;
                for (int q = 0; q < P.S; ++q)
                    s += __ldcg(P.ws + size_t(q) * sst + size_t(tile) * kTileRows + i % kTileRows);
                if (FUSE)
                    for (int q = 0; q < P.S; ++q)
                        su += __ldcg(P.ws + size_t(q) * sst + size_t(tile + 1) * kTileRows +
                                     i % kTileRows);
                store(tile, i % kTileRows, s, su);
            }
            named_sync(1, W * 32);
            for (int i = threadIdx.x; i < k; i += W * 32)
                if (flags[i])
                    tick[items[i]] = 0u;  // every slice of the item has been added
        }
    }

    __syncthreads();
    if (s_abort && threadIdx.x == 0) {
        // Let copies still in flight land before shared memory is released:
        // only the last NS issued slots can be outstanding.
        for (int i = s_issued - NS < 0 ? 0 : s_issued - NS; i < s_issued; ++i)
            mbar_wait_bounded(&full[i % NS], unsigned(i / NS) & 1u, 100000000ll);
    }
}

int env_m1_slices()
{
    const char *e = getenv("QMM_M1_S");
    return e ? atoi(e) : 0;
}

} // namespace

size_t m1_smem(int KS, int WS, int TS, int cap, int nslot, int sb_bytes)
{
    const int W = WS * TS;
    const size_t xn = sb_bytes == 210 ? 16 : 8;  // activation sums per super-block
    return size_t(nslot) * (size_t(W) * kTileRows * sb_bytes + 16) + size_t(KS) * 1024 + size_t(KS) * xn * 4 +
           size_t((KS + 3) & ~3) * 4 + size_t(WS) * cap * TS * kTileRows * 4 + size_t(cap) * 8 + 8;
}

int env_m1_warps()
{
    const char *e = getenv("QMM_M1_WARPS");
    return (e && atoi(e) == 8) ? 8 : kM1MaxWarps;
}

M1Plan plan_m1(int64_t T, int64_t NB, int sm_count, int force_S, int maxw, int sb_bytes,
               int min_ts, int upw)
{
    M1Plan p;
    if (maxw <= 0)
        maxw = env_m1_warps();
    maxw = maxw <= 8 ? 8 : kM1MaxWarps;
    // 8 consumer warps: half an SM, so that the next launch in the stream
    // can be resident beside this one; 16: the whole SM.
    const size_t budget = maxw <= 8 ? kM1SmemBudgetHalf : kM1SmemBudgetWhole;
    // K slices: the fewest (dividing NB) with at most 16 super-blocks each --
    // one pass, x laid out per CTA for 16 super-blocks at most: laying out a
    // long x in every CTA costs more than adding slices -- else the fewest
    // whose layout of x leaves two thirds of shared memory to the ring.
    // QMM_M1_S (or force_S) fixes S.
    const int forced = force_S > 0 ? force_S : env_m1_slices();
    // (WS, TS) for a slice of ks super-blocks: the most consumer warps that
    // still leave every SM an item, then the widest pass.
    // Q6_K (210-byte super-blocks): a TMA box spans 8 super-blocks (1680
    // bytes, the first whole multiple of 16 bytes), so passes are 8 wide.
    const bool q6 = sb_bytes == 210;
    auto shape = [&](int ks, int s_, int &ws_best, int &ts_best) {
        double best = -1.0;
        const int per = sm_count / s_ >= 1 ? sm_count / s_ : 1;
        for (int ws = (ks < maxw ? ks : maxw); ws >= 1; --ws) {
            if (ks % ws || (q6 && ws != 8))
                continue;
            for (int ts = min_ts > upw ? min_ts : upw; ts <= 8 && ws * ts <= maxw * upw; ts *= 2) {
                const int64_t items = (T + ts - 1) / ts;
                const double use = items >= per ? 1.0 : double(items) / per;
                const double score = ws * ts / upw * use;
                if (score > best + 1e-9) {
                    best = score;
                    ws_best = ws;
                    ts_best = ts;
                }
            }
        }
        return best;
    };
    int S = 0;
    if (forced > 0 && NB % forced == 0 && forced <= sm_count)
        S = forced;
    // K slices: among those with one pass (at most 16 super-blocks, laid out
    // per CTA -- laying out a long x in every CTA costs more than slices),
    // the most consumer warps, then the fewest slices; else the fewest whose
    // layout of x leaves two thirds of shared memory to the ring.
    double best = -1.0;
    for (int64_t cand = 1; S == 0 && cand <= NB && cand <= sm_count; ++cand) {
        if (NB % cand || NB / cand > maxw || size_t(NB / cand) * 1056 > budget / 3)
            continue;
        int ws = 0, ts = 0;
        const double sc = shape(int(NB / cand), int(cand), ws, ts);
        if (sc > best + 1e-9)
            best = sc;
    }
    for (int64_t cand = 1; S == 0 && best > 0 && cand <= NB && cand <= sm_count; ++cand) {
        if (NB % cand || NB / cand > maxw || size_t(NB / cand) * 1056 > budget / 3)
            continue;
        int ws = 0, ts = 0;
        if (shape(int(NB / cand), int(cand), ws, ts) >= best - 1e-9)
            S = int(cand);
    }
    for (int64_t cand = 1; S == 0 && cand <= NB && cand <= sm_count; ++cand)
        if (NB % cand == 0 && size_t(NB / cand) * 1056 <= budget / 3 && (!q6 || (NB / cand) % 8 == 0))
            S = int(cand);
    if (S == 0)
        return p;  // nslot == 0: not supported
    p.maxw = maxw;
    p.S = S;
    p.KS = int(NB / S);
    // Pass width WS (a divisor of KS, at most maxw) and tiles per item TS.
    if (shape(p.KS, S, p.WS, p.TS) < 0)
        return M1Plan();  // no pass width fits (Q6_K: KS not a multiple of 8)
    const int per_slice = sm_count / S >= 1 ? sm_count / S : 1;
    p.NP = p.KS / p.WS;
    p.upw = upw;
    p.W = p.WS * p.TS / upw;
    p.n_items = int((T + p.TS - 1) / p.TS);
    // One CTA per SM and slice; for very tall matrices more (several waves),
    // so that a CTA's share stays within kM1MaxShare items.
    p.G1 = per_slice;
    if ((p.n_items + p.G1 - 1) / p.G1 > kM1MaxShare)
        p.G1 = (p.n_items + kM1MaxShare - 1) / kM1MaxShare;
    if (p.G1 > p.n_items)
        p.G1 = p.n_items;
    const int avg = (p.n_items + p.G1 - 1) / p.G1;
    // Ring slots: as many as shared memory holds (at most 16) next to room
    // for twice a CTA's average share of items; if fewer than three slots
    // fit, the item room shrinks (never below one item over the average).
    p.cap = 2 * avg + 2;
    // QMM_M1_NSLOT caps the ring (a tuning knob)
    const char *en = getenv("QMM_M1_NSLOT");
    const int ns_max = (en && atoi(en) >= 2 && atoi(en) <= 16) ? atoi(en) : 16;
    auto slots = [&](int cap) {
        int ns = 0;
        while (ns < ns_max && m1_smem(p.KS, p.WS, p.TS, cap, ns + 1, sb_bytes) <= budget)
            ++ns;
        return ns;
    };
    int ns = slots(p.cap);
    while (ns < 3 && p.cap > avg + 1)
        ns = slots(--p.cap);
    if (ns < 2)
        return M1Plan();  // x's layout leaves no room for a ring: not supported
    p.nslot = ns;
    // Fixed items per CTA: the whole share (rounded up) when it fits the
    // ring, so that all of it is fetched before the previous kernel ends;
    // else three quarters of it.  The rest comes from the counter.
    p.F = avg * p.NP <= ns ? avg : (3 * p.n_items) / (4 * p.G1);
    if (p.F < 1)
        p.F = 1;
    p.slot_bytes = p.WS * p.TS * kTileRows * sb_bytes;  // units of the slot
    p.smem = m1_smem(p.KS, p.WS, p.TS, p.cap, ns, sb_bytes);
    p.ws_floats = S > 1 ? size_t(S) * size_t(T) * kTileRows : 0;
    p.tickets = size_t(2 * S) + (S > 1 ? size_t(p.n_items) : 0);
    return p;
}

cudaError_t launch_gemv_m1(const M1Args &a, const M1Plan &p, cudaStream_t s)
{
    M1Params P;
    memset(&P, 0, sizeof(P));
    int tiles = 0;
    for (int i = 0; i < a.nmat; ++i) {
        P.tmap[i] = *reinterpret_cast<const CUtensorMap *>(a.tmap[i]);
        tiles += int((a.rows[i] + kTileRows - 1) / kTileRows);
        P.tile_end[i] = tiles;
        P.rows[i] = int(a.rows[i]);
        P.y[i] = a.y[i];
    }
    for (int i = a.nmat; i < kMaxGroup; ++i)
        P.tile_end[i] = tiles;
    P.x = a.x;
    P.ws = a.ws;
    P.ctr = a.tickets;
    P.status = a.status;
    P.T = tiles;
    P.nmat = a.nmat;
    P.S = p.S;
    P.KS = p.KS;
    P.WS = p.WS;
    P.NP = p.NP;
    P.TS = p.TS;
    P.W = p.W;
    P.G1 = p.G1;
    P.n_items = p.n_items;
    P.F = p.F;
    P.cap = p.cap;
    P.nslot = p.nslot;
    P.slot_bytes = p.slot_bytes;
    // the fused pair runs the two-unit kernel, everything else the one-unit one
    if ((a.fuse_swiglu != 0) != (p.upw == 2) ||
        (a.fuse_swiglu && (a.nmat != 2 || a.rows[0] != a.rows[1] || p.TS % 2 != 0)))
        return cudaErrorInvalidValue;
    // All shared memory preferred, so that two half-SM CTAs (this launch
    // and the next) fit side by side.
    const bool two = p.upw == 2;
    const auto kern = a.fmt == QMM_Q5_K     ? (two ? gemv_m1_kernel<QMM_Q5_K, 2> : gemv_m1_kernel<QMM_Q5_K, 1>)
                      : a.fmt == QMM_Q6_K   ? (two ? gemv_m1_kernel<QMM_Q6_K, 2> : gemv_m1_kernel<QMM_Q6_K, 1>)
                      : a.fmt == QMM_IQ4_NL ? (two ? gemv_m1_kernel<QMM_IQ4_NL, 2> : gemv_m1_kernel<QMM_IQ4_NL, 1>)
                      : a.fmt == QMM_Q8_0   ? (two ? gemv_m1_kernel<QMM_Q8_0, 2> : gemv_m1_kernel<QMM_Q8_0, 1>)
                                            : (two ? gemv_m1_kernel<QMM_Q4_K, 2> : gemv_m1_kernel<QMM_Q4_K, 1>);
    cudaError_t e = func_smem(reinterpret_cast<const void *>(kern), p.smem, true);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(p.G1 * p.S));
    cfg.blockDim = dim3(unsigned((p.W + 1) * 32));
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return counted(cudaLaunchKernelEx(&cfg, kern, P));
}

} // namespace qmm
