// gemm_tc.cu -- Q4_K and Q8_0 prefill GEMM on the 5th-generation tensor cores
// (tcgen05.mma with the accumulators in tensor memory), dequantising the
// weights into shared memory on the way.
//
// The operation: "Frink Inference: the Rust alternative to llama.cpp",
// section "Where llama.cpp is still ahead" -- prompt processing (prefill),
// where many tokens go through every weight matrix at once, so the matmul is
// compute-bound rather than bandwidth-bound; and "Building a Rust Inference
// Engine That Matches Llama.cpp", "Where the wins came from" -- dequantise
// once per weight, in fast memory, not as a separate pass over a
// full-precision copy.
//
//   Y[m][n] = sum_k bf16(w[n][k]) * X[m][k]     (fp32 accumulation)
//
// bf16(w) is the exact Q4_K weight d*sc*q - dmin*m rounded to fp32 and then
// to bfloat16 (nearest even), the same values qmm_dequantize_bf16 returns.
//
// Tiling.  One CTA tile is 256 tokens x 256 weight rows: the tokens are the
// MMA's M side (A operand, TMEM lanes; two halves of 128) and the weight rows
// its N side (B operand, TMEM columns), so each dequantised weight feeds 256
// tokens and each epilogue thread owns one token's row of Y.  K advances in
// stages of 64 (one 128-byte swizzle row of bf16):
//   A    256 x 64 bf16 of X, one TMA box, 128-byte swizzle         (32 KB)
//   nib  the 32 nibble bytes of this 64-weight chunk, 256 rows      (8 KB)
//   B    256 x 64 bf16 weights, written by the dequant warps in the
//        same swizzled K-major layout                               (32 KB)
// and once per super-block the rows' 16-byte headers (4 KB, two slots).
// Eight m128 n256 k16 MMAs per stage (four K steps x two token halves)
// accumulate into two 256-column TMEM accumulators (all 512 columns).
// Tiles are spread over a persistent grid.
//
// Three rings of their own depth.  A stage's X is needed from its copy to
// its MMAs, its raw weight bytes from their copy until the dequant warps
// have written the stage's B, its bf16 B from the dequantisation to the
// MMAs.  One ring of (X, raw, B) stages would hold every buffer for the copy
// latency plus the dequantisation plus the MMAs, and three such stages are
// all that shared memory takes; separate rings hold each buffer only for its
// own part (X: copy + MMAs; raw: copy + dequantisation; B: dequantisation +
// MMAs), so the X ring can be deeper, the raw bytes run ahead of the X
// copies and the dequantisation overlaps the MMAs of the previous stage.  The producer
// feeds the X and raw rings as two independent streams (polling both
// rings' free slots), so neither waits behind the other.
//
// Warp roles (576 threads):
//   warp 0        TMA producer (one lane)
//   warp 1        TMEM allocation and MMA issue (one lane)
//   warps 2..9    epilogue: TMEM -> registers -> Y.  Warp w reads TMEM lanes
//                 32*(w%4) .. +31 (the quarter it may access) of token half
//                 (w-2)/4.
//   warps 10..17  dequantisation, one weight row per thread
//
// Every pipeline wait is bounded.  A wait that runs out records the timeout
// in the status word and raises a CTA-wide abort flag; every role then leaves
// its loop, the copies and MMAs already issued are waited for (again with a
// limit), and the tensor memory is released before the CTA exits.
#include <cstring>

#include <cuda.h>

#include "qmm_device.cuh"
#include "qmm_internal.h"
#include "tcgen05.cuh"

namespace qmm {

namespace {

using namespace t5;

constexpr int kRows = 256;            // weight rows per tile (MMA N)
constexpr int kBBytes = kRows * 128;  // 32768
constexpr int kNibBytes = kRows * 32; // 8192
constexpr int kHdrBytes = kRows * 16; // 4096
constexpr int kHdrSlots = 2;
constexpr int kEpiStage = 32 * 32 * 4;               // one 32-token x 32-column fp32 chunk
constexpr size_t kEpiStageBytes = 8 * kEpiStage;     // one per epilogue warp
constexpr int kThreads = 576;
constexpr int kEpiWarp0 = 2;
constexpr int kDequantWarp0 = 10;
constexpr int kMaxKSplit = 16;

// Token tiles of 256 (two MMAs of M = 128 per K step into both 256-column
// TMEM accumulators) or of 128 (one MMA, one accumulator) for problems whose
// 256-token tiles would not fill the SMs.
// Weight bytes staged per 64-weight K step and 256 rows: Q4_K the chunk's 32
// nibble bytes (its 16-byte header separately, once per super-block); Q8_0
// the chunk's two 34-byte blocks, fetched as the 80-byte window that starts
// at the 16-byte boundary at or below them (a TMA box must start there).
constexpr int kQ80Window = 80;
template <int FMT> constexpr int kRawBytes = FMT == QMM_Q4_K ? kNibBytes : kRows * kQ80Window;

// Ring depths: NX stages of X, NB of bf16 B, NR of raw weight bytes.
template <int TOK, int FMT, int NX, int NB, int NR>
struct TileCfg {
    static constexpr int kTok = TOK;
    static constexpr int kHalves = TOK / 128;           // MMAs of M = 128 per K step
    static constexpr int kABytes = TOK * 128;
    static constexpr int kRaw = kRawBytes<FMT>;
    static constexpr int kHdr = FMT == QMM_Q4_K ? kHdrSlots : 0;
    static constexpr uint32_t kTmemCols = uint32_t(kHalves) * 256;
    static constexpr int kBars = 2 * NX + 2 * NB + 2 * NR + 2 * kHdrSlots + 3;
    static constexpr size_t kSmemBytes = 1024 /* alignment slack */ + size_t(NX) * kABytes +
                                         size_t(NB) * kBBytes + size_t(NR) * kRaw +
                                         size_t(kHdr) * kHdrBytes + kEpiStageBytes + size_t(kBars) * 8;
    static_assert(kSmemBytes <= 232448, "shared memory per block");
    static_assert(NR <= 8, "two header slots: the raw stream runs at most NR stages ahead");
};

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulate, A and B
// bf16, both K-major, N = 256 (bits 17-22 hold N/8), M = 128 (bits 24-28
// hold M/16).
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(kRows >> 3) << 17) |
                            (uint32_t(128 >> 4) << 24);

struct GemmParams {
    CUtensorMap tm_x;                   // X [M][K] bf16, box 64 x 256, 128-byte swizzle
    CUtensorMap tm_hdr[kGemmMaxGroup];  // weight bytes [N_i][row_bytes] u8, box 16 x 256
    CUtensorMap tm_nib[kGemmMaxGroup];  // weight bytes, box 32 x 256 (Q8_0: 80 x 256)
    CUtensorMap tm_y[kGemmMaxGroup];    // Y_i [M][N_i] fp32, box 32 x 32, 128-byte swizzle
    CUtensorMap tm_ws;                  // partials [ksplit][M][Ntot] fp32, box 32 x 32 x 1
    float *y[kGemmMaxGroup];            // [M][N_i]
    int n_rows[kGemmMaxGroup];          // N_i
    int rt_end[kGemmMaxGroup];          // cumulative 256-row tiles
    int col_off[kGemmMaxGroup];         // first column of matrix i in the partials
    int nmat;
    int Ntot;                           // sum of N_i
    float *ws;           // split-K partials [ksplit][M][Ntot] (ksplit > 1)
    int M, K;
    int tok_tiles, tiles;
    int ksplit;          // K slices of each tail tile (at most K / 256)
    int full_units;      // tiles [0, full_units) run whole, one unit each
    int units;           // full_units + (tiles - full_units) * ksplit
    int vec_store;       // Y rows 16-byte aligned: store float4
    int tma_store;       // tm_y (and tm_ws when split) are valid: bulk-store whole chunks
    unsigned *status;
};

// Global 256-row tile -> (matrix of the group, first row within it).
__device__ __forceinline__ void matrix_row_tile(const GemmParams &P, int grt, int &mi, int &row0)
{
    mi = 0;
#pragma unroll
    for (int i = 0; i < kGemmMaxGroup - 1; ++i)
        if (i < P.nmat - 1 && grt >= P.rt_end[i])
            mi = i + 1;
    row0 = (grt - (mi == 0 ? 0 : P.rt_end[mi - 1])) * kRows;
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t accumulate)
{
    mma_f16(d_tmem, adesc, bdesc, kIdesc, accumulate);
}

// Four weights of one nibble lane of word v (mask 0x0F0F0F0F: the low
// nibbles, values q; mask 0xF0F0F0F0: the high nibbles, values 16q) as two
// bf16 pairs of RN_fp32(a*q - b); `as` is a (or a/16 for the high nibbles).
__device__ __forceinline__ void dequant4(uint32_t v, float as, float b, uint32_t &p0, uint32_t &p1)
{
    const float2 magic = make_float2(-8388608.f, -8388608.f);
    const float2 A = make_float2(as, as), B = make_float2(-b, -b);
    float2 f0 = make_float2(byte_magic(v, 0), byte_magic(v, 1));
    float2 f1 = make_float2(byte_magic(v, 2), byte_magic(v, 3));
    f0 = __fadd2_rn(f0, magic);  // q (or 16q), exact
    f1 = __fadd2_rn(f1, magic);
    f0 = __ffma2_rn(f0, A, B);   // RN(a*q - b)
    f1 = __ffma2_rn(f1, A, B);
    p0 = cvt_bf16x2(f0.x, f0.y);
    p1 = cvt_bf16x2(f1.x, f1.y);
}

// Four Q8_0 weights (int8 bytes of v) as two bf16 pairs of RN(d*q); d*q is
// exact in fp32.
__device__ __forceinline__ void dequant4_q8(uint32_t v, float d, uint32_t &p0, uint32_t &p1)
{
    const float2 off = make_float2(-8388736.f, -8388736.f);  // -(2^23 + 128)
    const float2 D = make_float2(d, d);
    const uint32_t u = v ^ 0x80808080u;  // q + 128 in each byte
    float2 f0 = make_float2(byte_magic(u, 0), byte_magic(u, 1));
    float2 f1 = make_float2(byte_magic(u, 2), byte_magic(u, 3));
    f0 = __fmul2_rn(__fadd2_rn(f0, off), D);
    f1 = __fmul2_rn(__fadd2_rn(f1, off), D);
    p0 = cvt_bf16x2(f0.x, f0.y);
    p1 = cvt_bf16x2(f1.x, f1.y);
}

template <int TOK, int FMT, int NX, int NB, int NR>
__global__ void __launch_bounds__(kThreads, 1) gemm_q4k_kernel(const __grid_constant__ GemmParams P)
{
    using C = TileCfg<TOK, FMT, NX, NB, NR>;
    constexpr int kRaw = C::kRaw, kHS = kHdrSlots;
    constexpr int kTok = C::kTok, kABytes = C::kABytes;
    constexpr uint32_t kTmemCols = C::kTmemCols;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base_u32 = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_u32 - smem_u32(smem_raw));
    uint8_t *sA = base;                                  // [NX][TOK x 128 B]
    uint8_t *sB = sA + NX * kABytes;                     // [NB][32 KB]
    uint8_t *sRaw = sB + NB * kBBytes;                   // [NR][kRaw]
    uint8_t *sHdr = sRaw + NR * kRaw;                    // [kHdr][4 KB]
    uint8_t *sEpi = sHdr + C::kHdr * kHdrBytes;          // [8 epilogue warps][4 KB], 1024-aligned
    uint64_t *bars = reinterpret_cast<uint64_t *>(sEpi + kEpiStageBytes);
    uint64_t *xfull = bars;                 // X landed                (tx)
    uint64_t *xempty = xfull + NX;          // MMAs of the X slot done (commit)
    uint64_t *bready = xempty + NX;         // B written               (8 dequant warps)
    uint64_t *bempty = bready + NB;         // MMAs of the B slot done (commit)
    uint64_t *rfull = bempty + NB;          // raw bytes landed        (tx)
    uint64_t *rempty = rfull + NR;          // raw bytes used          (8 dequant warps)
    uint64_t *hfull = rempty + NR;          // headers landed          (tx)
    uint64_t *hempty = hfull + kHS;         // headers used            (8 dequant warps)
    uint64_t *accfull = hempty + kHS;       // accumulators complete   (commit)
    uint64_t *accempty = accfull + 1;       // accumulators drained    (8 epilogue warps)
    uint64_t *drain = accempty + 1;         // final MMA drain         (commit)
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sb_n = P.K / 256;
    // Unit un: a whole tile (un < full_units) or K slice `kslice` of one of
    // the tail tiles: super-blocks [kslice * n / ks, (kslice + 1) * n / ks)
    // of the n = K / 256 (slices differ by at most one super-block).
    auto unit_of = [&](int un, int &t, int &kslice, int &sb0, int &sb_u) {
        if (un < P.full_units) {
            t = un;
            kslice = 0;
            sb0 = 0;
            sb_u = sb_n;
        } else {
            const int v = un - P.full_units;
            t = P.full_units + v / P.ksplit;
            kslice = v - (v / P.ksplit) * P.ksplit;
            sb0 = kslice * sb_n / P.ksplit;
            sb_u = (kslice + 1) * sb_n / P.ksplit - sb0;
        }
    };

    // The descriptors of the first copies and stores, fetched while the
    // previous kernel drains.
    if (threadIdx.x == 32 * kEpiWarp0)
        prefetch_tmap(&P.tm_x);
    if (threadIdx.x >= 32 * kEpiWarp0 + 1 && threadIdx.x < 32 * kEpiWarp0 + 1 + P.nmat) {
        const int i = int(threadIdx.x) - 32 * kEpiWarp0 - 1;
        prefetch_tmap(&P.tm_nib[i]);
        if (FMT == QMM_Q4_K)
            prefetch_tmap(&P.tm_hdr[i]);
        if (P.tma_store)
            prefetch_tmap(&P.tm_y[i]);
    }
    if (threadIdx.x == 32 * kEpiWarp0 + 8 && P.tma_store && P.ksplit > 1)
        prefetch_tmap(&P.tm_ws);
    if (threadIdx.x == 0) {
        for (int s = 0; s < NX; ++s) {
            mbar_init(&xfull[s], 1);
            mbar_init(&xempty[s], 1);
        }
        for (int s = 0; s < NB; ++s) {
            mbar_init(&bready[s], 8);
            mbar_init(&bempty[s], 1);
        }
        for (int s = 0; s < NR; ++s) {
            mbar_init(&rfull[s], 1);
            mbar_init(&rempty[s], 8);
        }
        for (int h = 0; h < kHS; ++h) {
            mbar_init(&hfull[h], 1);
            mbar_init(&hempty[h], 8);
        }
        mbar_init(accfull, 1);
        mbar_init(accempty, 8);
        mbar_init(drain, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_base_sh)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    // X, Y and the split-K scratch belong to earlier kernels until their
    // dependency wait: the producer waits before its first X copy and the
    // epilogue before its first store.  The weights are the handle's, fixed
    // before any call, so their ring fills (and the dequant warps start)
    // while the previous kernel drains; the MMA and dequant warps touch only
    // shared and tensor memory.
    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            // Two cursors over this CTA's stages (units blockIdx.x, +grid, ...,
            // each a run of 64-wide K steps): the X stream and the raw stream.
            struct Cursor {
                int un, ks, ks_end, tok0, mi, row0;
            };
            auto seek = [&](Cursor &c, int un) {
                c.un = un;
                if (un >= P.units)
                    return;
                int t, kslice, sb0, sb_u;
                unit_of(un, t, kslice, sb0, sb_u);
                matrix_row_tile(P, t / P.tok_tiles, c.mi, c.row0);
                c.tok0 = (t % P.tok_tiles) * kTok;
                c.ks = 4 * sb0;
                c.ks_end = 4 * (sb0 + sb_u);
            };
            auto step = [&](Cursor &c) {
                if (++c.ks == c.ks_end)
                    seek(c, c.un + int(gridDim.x));
            };
            Cursor cx, cr;
            seek(cx, blockIdx.x);
            seek(cr, blockIdx.x);
            int ix = 0, ir = 0, hit = 0;  // stages / super-blocks issued per stream
            // Is the raw slot of stage ir (and, at a super-block's first
            // chunk, a header slot) free?
            auto raw_free = [&]() {
                const int s = ir % NR, c = cr.ks & 3;
                const bool with_hdr = FMT == QMM_Q4_K && c == 0;
                const int h = hit % kHS;
                return (ir < NR || mbar_test_wait(&rempty[s], unsigned(ir / NR - 1) & 1u)) &&
                       (!with_hdr || hit < kHS ||
                        mbar_test_wait(&hempty[h], unsigned(hit / kHS - 1) & 1u));
            };
            auto issue_raw = [&]() {
                const int s = ir % NR, sb = cr.ks >> 2, c = cr.ks & 3;
                if (FMT == QMM_Q4_K && c == 0) {
                    const int h = hit % kHS;
                    mbar_arrive_expect_tx(&hfull[h], kHdrBytes);
                    tma_2d(sHdr + h * kHdrBytes, &P.tm_hdr[cr.mi], sb * 144, cr.row0, &hfull[h]);
                    ++hit;
                }
                // Q8_0: the chunk's blocks sit at 272 sb + 68 c of the row
                const int xoff = FMT == QMM_Q8_0 ? 272 * sb + ((68 * c) & ~15) : sb * 144 + 16 + 32 * c;
                mbar_arrive_expect_tx(&rfull[s], kRaw);
                tma_2d(sRaw + s * kRaw, &P.tm_nib[cr.mi], xoff, cr.row0, &rfull[s]);
                ++ir;
                step(cr);
            };
            // The weights first: the raw ring's free slots before the wait.
            while (cr.un < P.units && ir < NR && raw_free())
                issue_raw();
            pdl_wait();
            long long idle0 = clock64();
            while (!abort_flag && (cx.un < P.units || cr.un < P.units)) {
                bool moved = false;
                // X of stage ix into slot ix % NX, once the MMAs of its previous
                // stage there are done.
                if (cx.un < P.units &&
                    (ix < NX || mbar_test_wait(&xempty[ix % NX], unsigned(ix / NX - 1) & 1u))) {
                    const int s = ix % NX;
                    mbar_arrive_expect_tx(&xfull[s], kABytes);
                    tma_2d(sA + s * kABytes, &P.tm_x, cx.ks * 64, cx.tok0, &xfull[s]);
                    ++ix;
                    step(cx);
                    moved = true;
                }
                // Raw bytes of stage ir (and, at a super-block's first chunk,
                // its headers), once the dequant warps hold the previous ones.
                if (cr.un < P.units && raw_free())
                    issue_raw(), moved = true;
                if (moved) {
                    idle0 = clock64();
                } else if (clock64() - idle0 > kWaitBudgetCycles) {
                    atomicOr(P.status, kStatusTimeoutBit);
                    abort_flag = 1;
                } else {
                    __nanosleep(32);
                }
            }
            // Copies still in flight must land before the CTA exits: wait for
            // the last phase of every slot that was used (bounded).
            for (int s = 0; s < NX && s < ix; ++s)
                mbar_wait_bounded(&xfull[s], unsigned((ix - 1 - s) / NX) & 1u, 200000000ll);
            for (int s = 0; s < NR && s < ir; ++s)
                mbar_wait_bounded(&rfull[s], unsigned((ir - 1 - s) / NR) & 1u, 200000000ll);
            for (int h = 0; h < kHS && h < hit; ++h)
                mbar_wait_bounded(&hfull[h], unsigned((hit - 1 - h) / kHS) & 1u, 200000000ll);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issue
        if (lane == 0) {
            int it = 0, lt = 0;
            for (int un = blockIdx.x; un < P.units && !abort_flag; un += gridDim.x, ++lt) {
                if (lt >= 1 && !wait_phase(accempty, unsigned(lt - 1) & 1u, &abort_flag, P.status))
                    break;
                tc_fence_after();
                bool ok = true;
                int t_, ksl_, sb0_, sb_u;
                unit_of(un, t_, ksl_, sb0_, sb_u);
                for (int ks = 0; ks < 4 * sb_u; ++ks, ++it) {
                    const int sx = it % NX, sbf = it % NB;
                    if (!wait_phase(&xfull[sx], unsigned(it / NX) & 1u, &abort_flag, P.status) ||
                        !wait_phase(&bready[sbf], unsigned(it / NB) & 1u, &abort_flag, P.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + sx * kABytes), b0 = smem_u32(sB + sbf * kBBytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bd = sw128_desc(b0 + 32 * kk);
                        const uint32_t acc = (ks | kk) != 0 ? 1u : 0u;
#pragma unroll
                        for (int h = 0; h < C::kHalves; ++h)
                            mma_bf16(tmem + uint32_t(h * kRows), sw128_desc(a0 + h * 16384 + 32 * kk),
                                     bd, acc);
                    }
                    mma_commit(&xempty[sx]);
                    mma_commit(&bempty[sbf]);
                }
                if (!ok)
                    break;
                mma_commit(accfull);
            }
            // Every MMA issued has finished once this commit arrives.
            mma_commit(drain);
            mbar_wait_bounded(drain, 0u, 200000000ll);
        }
    } else if (warp < kDequantWarp0) {
        // ---------------------------------------------------------- epilogue
        // A warp's 32 tokens x 32 columns per chunk: TMEM -> registers -> its
        // staging buffer (row = token, 128-byte swizzle) -> one bulk tensor
        // store into Y (or the partials).  The accumulators are free once the
        // last chunk is in registers; the stores complete in the background.
        // Chunks a store cannot take (Y not 16-byte aligned, a partial
        // 32-column piece) are written by the threads themselves.
        pdl_wait();  // Y and the partials belong to earlier kernels until here
        const int quarter = warp & 3;
        const int eh = (warp - kEpiWarp0) >> 2;  // 256-token tiles: token half; 128: column half
        const int tok_in_tile = (C::kHalves == 2 ? eh * 128 : 0) + quarter * 32 + lane;
        constexpr int kCols = C::kHalves == 2 ? kRows : kRows / 2;  // columns this warp drains
        const int col0 = C::kHalves == 2 ? 0 : eh * (kRows / 2);
        uint8_t *stage = sEpi + (warp - kEpiWarp0) * kEpiStage;
        uint8_t *srow = stage + lane * 128;
        const uint32_t sw = uint32_t(lane & 7);
        bool pending = false;  // lane 0 has a bulk store that may still read the buffer
        int lt = 0;
        for (int un = blockIdx.x; un < P.units; un += gridDim.x, ++lt) {
            if (!wait_phase(accfull, unsigned(lt) & 1u, &abort_flag, P.status))
                break;
            tc_fence_after();
            int t, kslice, sb0_, sb_u_;
            unit_of(un, t, kslice, sb0_, sb_u_);
            const bool split = un >= P.full_units && P.ksplit > 1;
            const int tok = (t % P.tok_tiles) * kTok + tok_in_tile;
            const int tok_w = tok - lane;  // the warp's first token
            int mi, row0;
            matrix_row_tile(P, t / P.tok_tiles, mi, row0);
            const int Nm = P.n_rows[mi];
            // With K split, slice k writes its partial product to ws[k] (the
            // group's matrices side by side, Ntot columns); a reduction
            // kernel adds the slices in order.
            float *yrow = split ? P.ws + (size_t(kslice) * size_t(P.M) + tok) * P.Ntot + P.col_off[mi]
                                : P.y[mi] + int64_t(tok) * Nm;
            const uint32_t taddr = tmem + (uint32_t(quarter * 32) << 16) +
                                   uint32_t(C::kHalves == 2 ? eh * kRows : col0);
#pragma unroll 1
            for (int ch = 0; ch < kCols / 32; ++ch) {
                uint32_t r[32];
                tmem_ld16(taddr + uint32_t(ch * 32), *reinterpret_cast<uint32_t(*)[16]>(r));
                tmem_ld16(taddr + uint32_t(ch * 32 + 16), *reinterpret_cast<uint32_t(*)[16]>(r + 16));
                tmem_ld_wait();
                const int n0 = row0 + col0 + ch * 32;
                if (P.tma_store && n0 + 32 <= Nm) {
                    if (tok_w >= P.M)
                        continue;
                    if (pending && lane == 0)
                        bulk_wait_read();  // the previous chunk has left the buffer
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<uint4 *>(srow + ((uint32_t(j) ^ sw) << 4)) =
                            make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
                    fence_proxy_async_smem();  // the bulk store reads the buffer through the async proxy
                    __syncwarp();
                    if (lane == 0) {
                        if (split)
                            tma_store_3d(&P.tm_ws, stage, P.col_off[mi] + n0, tok_w, kslice);
                        else
                            tma_store_2d(&P.tm_y[mi], stage, n0, tok_w);
                        bulk_commit();
                        pending = true;
                    }
                } else if (tok < P.M) {
                    if (P.vec_store && n0 + 32 <= Nm) {
                        float4 *dst = reinterpret_cast<float4 *>(yrow + n0);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                                 __uint_as_float(r[4 * i + 2]),
                                                 __uint_as_float(r[4 * i + 3]));
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (n0 + i < Nm)
                                yrow[n0 + i] = __uint_as_float(r[i]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(accempty);  // the accumulators are free for the next unit
        }
        if (pending && lane == 0)
            bulk_wait_all();  // the stores are complete before the CTA exits
    } else {
        // ---------------------------------------------------------- dequantisation
        // Per stage: load the raw bytes, wait for the B slot (the MMAs of its
        // previous stage), write the bf16 weights, then free the B slot's
        // contents to the MMA and the raw slot to the producer.  The raw slot
        // is freed only after the stores that use its bytes, so the order of
        // the reads and the release rests on a data dependency, not on how
        // the loads are scheduled.
        const int r = (warp - kDequantWarp0) * 32 + lane;  // weight row within the tile
        const uint32_t swz = uint32_t(r & 7);
        int it = 0, hit = 0;
        bool ok = true;
        if constexpr (FMT == QMM_Q8_0) {
            for (int un = blockIdx.x; un < P.units && ok; un += gridDim.x) {
                int t_, ksl_, sb0, sb_u;
                unit_of(un, t_, ksl_, sb0, sb_u);
                for (int ks = 4 * sb0; ks < 4 * (sb0 + sb_u); ++ks, ++it) {
                    const int s = it % NR, sbf = it % NB;
                    if (!wait_phase(&rfull[s], unsigned(it / NR) & 1u, &abort_flag, P.status)) {
                        ok = false;
                        break;
                    }
                    // this row's two blocks: [d0][32 q][d1][32 q] from byte
                    // (68 c) mod 16 of its window -- 17 aligned words
                    const uint32_t *wd = reinterpret_cast<const uint32_t *>(
                        sRaw + s * kRaw + r * kQ80Window + ((68 * (ks & 3)) & 15));
                    uint32_t W[17];
#pragma unroll
                    for (int i = 0; i < 17; ++i)
                        W[i] = wd[i];
                    if (it >= NB &&
                        !wait_phase(&bempty[sbf], unsigned(it / NB - 1) & 1u, &abort_flag, P.status)) {
                        ok = false;
                        break;
                    }
                    fence_proxy_async_smem();  // the slot's MMA reads (async proxy) before these writes
                    const float d0 = __half2float(__ushort_as_half((unsigned short)(W[0] & 0xffffu)));
                    const float d1 = __half2float(__ushort_as_half((unsigned short)(W[8] >> 16)));
                    uint8_t *brow = sB + sbf * kBBytes + r * 128;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {  // 16-byte chunk j: weights 8j .. 8j+7
                        uint32_t v0, v1;
                        if (j < 4) {  // block 0: codes at bytes 2..33 (2-byte offset)
                            v0 = __byte_perm(W[2 * j], W[2 * j + 1], 0x5432u);
                            v1 = __byte_perm(W[2 * j + 1], W[2 * j + 2], 0x5432u);
                        } else {      // block 1: codes at bytes 36..67 (aligned)
                            v0 = W[9 + 2 * (j - 4)];
                            v1 = W[10 + 2 * (j - 4)];
                        }
                        uint32_t p[4];
                        dequant4_q8(v0, j < 4 ? d0 : d1, p[0], p[1]);
                        dequant4_q8(v1, j < 4 ? d0 : d1, p[2], p[3]);
                        *reinterpret_cast<uint4 *>(brow + ((uint32_t(j) ^ swz) << 4)) =
                            make_uint4(p[0], p[1], p[2], p[3]);
                    }
                    fence_proxy_async_smem();  // the MMA reads B through the async proxy
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&bready[sbf]);
                        mbar_arrive(&rempty[s]);  // B was computed from them: the raw bytes are free
                    }
                }
            }
        }
        for (int un = blockIdx.x; un < P.units && ok && FMT == QMM_Q4_K; un += gridDim.x) {
            int t_, ksl_, sb0, sb_u;
            unit_of(un, t_, ksl_, sb0, sb_u);
            for (int sb = sb0; sb < sb0 + sb_u && ok; ++sb, ++hit) {
                const int h = hit % kHS;
                if (!wait_phase(&hfull[h], unsigned(hit / kHS) & 1u, &abort_flag, P.status)) {
                    ok = false;
                    break;
                }
                const uint4 hd = *reinterpret_cast<const uint4 *>(sHdr + h * kHdrBytes + r * 16);
                const float2 dd = half2_bits_to_float2(hd.x);
                for (int c = 0; c < 4; ++c, ++it) {
                    const int s = it % NR, sbf = it % NB;
                    if (!wait_phase(&rfull[s], unsigned(it / NR) & 1u, &abort_flag, P.status)) {
                        ok = false;
                        break;
                    }
                    const uint8_t *nib = sRaw + s * kRaw + r * 32;
                    const uint4 n0 = *reinterpret_cast<const uint4 *>(nib);
                    const uint4 n1 = *reinterpret_cast<const uint4 *>(nib + 16);
                    if (it >= NB &&
                        !wait_phase(&bempty[sbf], unsigned(it / NB - 1) & 1u, &abort_flag, P.status)) {
                        ok = false;
                        break;
                    }
                    fence_proxy_async_smem();  // the slot's MMA reads (async proxy) before these writes
                    uint32_t sc_lo, m_lo, sc_hi, m_hi;
                    scale_min(hd.y, hd.z, hd.w, 2 * c, sc_lo, m_lo);
                    scale_min(hd.y, hd.z, hd.w, 2 * c + 1, sc_hi, m_hi);
                    const float a_lo = dd.x * float(sc_lo), b_lo = dd.y * float(m_lo);
                    const float a_hi16 = dd.x * float(sc_hi) * 0.0625f, b_hi = dd.y * float(m_hi);
                    const uint32_t w[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
                    uint8_t *brow = sB + sbf * kBBytes + r * 128;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {  // chunks j (low nibbles) and j + 4 (high)
                        uint32_t p[4], q[4];
                        dequant4(w[2 * j] & 0x0F0F0F0Fu, a_lo, b_lo, p[0], p[1]);
                        dequant4(w[2 * j + 1] & 0x0F0F0F0Fu, a_lo, b_lo, p[2], p[3]);
                        dequant4(w[2 * j] & 0xF0F0F0F0u, a_hi16, b_hi, q[0], q[1]);
                        dequant4(w[2 * j + 1] & 0xF0F0F0F0u, a_hi16, b_hi, q[2], q[3]);
                        *reinterpret_cast<uint4 *>(brow + ((uint32_t(j) ^ swz) << 4)) =
                            make_uint4(p[0], p[1], p[2], p[3]);
                        *reinterpret_cast<uint4 *>(brow + ((uint32_t(j + 4) ^ swz) << 4)) =
                            make_uint4(q[0], q[1], q[2], q[3]);
                    }
                    fence_proxy_async_smem();  // the MMA reads B through the async proxy
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&bready[sbf]);
                        // B was computed from the raw bytes (and, by the last
                        // chunk, from every header word): both slots are free
                        mbar_arrive(&rempty[s]);
                        if (c == 3)
                            mbar_arrive(&hempty[h]);
                    }
                }
            }
        }
    }

    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

struct ReduceParams {
    float *y[kGemmMaxGroup];
    int n_rows[kGemmMaxGroup];
    int col_off[kGemmMaxGroup];
    int rt_end[kGemmMaxGroup];
    int nmat, Ntot, M, ks;
    int tok, tok_tiles, first_tail, n_tail;  // token tile height; tail tiles [first_tail, +n_tail)
    int vec;                            // every N_i % 4 == 0 and every Y 16-byte aligned
    const float *ws;
};

// For every tail tile (split in K): y_i[m][c] = ws[0][m][off_i + c] + ... +
// ws[ks-1][m][off_i + c], in slice order.  Four columns per thread (a tile
// is 256 wide and 16-byte aligned in the partials when every N_i % 4 == 0;
// otherwise the columns are handled one by one).
__global__ void splitk_reduce_kernel(const __grid_constant__ ReduceParams R)
{
    pdl_wait();
    pdl_launch_dependents();
    const int64_t plane = int64_t(R.M) * R.Ntot;
    const int64_t per_tile = int64_t(R.tok) * (kRows / 4);
    const int64_t n = int64_t(R.n_tail) * per_tile;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int tt = int(i / per_tile);
        const int rem = int(i - int64_t(tt) * per_tile);
        const int t = R.first_tail + tt;
        const int tok = (t % R.tok_tiles) * R.tok + rem / (kRows / 4);
        const int grt = t / R.tok_tiles;
        int mi = 0;
#pragma unroll
        for (int j = 0; j < kGemmMaxGroup - 1; ++j)
            if (j < R.nmat - 1 && grt >= R.rt_end[j])
                mi = j + 1;
        const int row = (grt - (mi == 0 ? 0 : R.rt_end[mi - 1])) * kRows + (rem % (kRows / 4)) * 4;
        if (tok >= R.M)
            continue;
        const int64_t e = int64_t(tok) * R.Ntot + R.col_off[mi] + row;
        float *dst = R.y[mi] + int64_t(tok) * R.n_rows[mi] + row;
        if (R.vec && row + 4 <= R.n_rows[mi]) {
            // slice order; the running sum keeps the registers (and so the
            // occupancy that hides the loads' latency) low
            float4 acc = __ldcs(reinterpret_cast<const float4 *>(R.ws + e));
#pragma unroll 4
            for (int k = 1; k < R.ks; ++k) {
                const float4 v = __ldcs(reinterpret_cast<const float4 *>(R.ws + k * plane + e));
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            *reinterpret_cast<float4 *>(dst) = acc;
        } else {
            for (int c = 0; c < 4 && row + c < R.n_rows[mi]; ++c) {
                float acc = __ldcs(R.ws + e + c);
                for (int k = 1; k < R.ks; ++k)
                    acc += __ldcs(R.ws + k * plane + e + c);
                dst[c] = acc;
            }
        }
    }
}

// The kernel instance and its shared memory for a token tile and format.
// Ring depths (NX, NB, NR) fill the 227 KB of shared memory beside the
// epilogue's 32 KB of staging; QMM_GEMM_RINGS selects one of the
// alternatives kept for Q4_K (1 or 2) in place of the default (0).
using GemmKernel = decltype(&gemm_q4k_kernel<256, QMM_Q4_K, 3, 2, 3>);
struct GemmInstance {
    GemmKernel fn;
    size_t smem;
};

template <int TOK, int FMT, int NX, int NB, int NR>
GemmInstance instance()
{
    return {gemm_q4k_kernel<TOK, FMT, NX, NB, NR>, TileCfg<TOK, FMT, NX, NB, NR>::kSmemBytes};
}

GemmInstance pick_gemm(int tok, int fmt)
{
    int v = 0;
    if (const char *e = getenv("QMM_GEMM_RINGS"))
        v = atoi(e);
    if (fmt == QMM_Q8_0)
        return tok == 128 ? instance<128, QMM_Q8_0, 4, 2, 3>() : instance<256, QMM_Q8_0, 2, 2, 3>();
    if (tok == 128)
        return v == 1   ? instance<128, QMM_Q4_K, 5, 2, 4>()
               : v == 2 ? instance<128, QMM_Q4_K, 6, 2, 3>()
                        : instance<128, QMM_Q4_K, 4, 3, 3>();
    return v == 1   ? instance<256, QMM_Q4_K, 2, 3, 3>()
           : v == 2 ? instance<256, QMM_Q4_K, 2, 2, 6>()
                    : instance<256, QMM_Q4_K, 3, 2, 3>();
}

} // namespace

size_t gemm_q4k_smem(int tok, int fmt)
{
    return pick_gemm(tok, fmt).smem;
}

int gemm_q4k_tiles(int64_t M, int64_t N, int tok)
{
    return int((M + tok - 1) / tok) * int((N + kRows - 1) / kRows);
}

// How to cut the work into units, from a time model: a CTA spends about
// 3.7 us per super-block of a 256 x 256 tile and runs its units one after the
// other (one CTA per SM).  Whole tiles fill full waves; the tiles of the last,
// partial wave (all tiles when there are fewer than the SMs) are split in K
// into `ksplit` slices (at most 16 and at most K/256; the super-blocks are
// shared out as evenly as they go, so the longest slice takes the ceiling),
// which costs writing and re-reading their fp32 partials at about 5 TB/s.
// The count with the least estimated time wins (1 = no split).
// QMM_GEMM_KSPLIT forces a value (at most K/256); then every tile is split.
GemmSplit gemm_q4k_split(int tiles, int tok, int64_t K, int sm_count)
{
    const int sb = int(K / 256);
    GemmSplit g;
    g.full = tiles;
    g.ksplit = 1;
    if (const char *e = getenv("QMM_GEMM_KSPLIT")) {
        const int f = atoi(e);
        if (f >= 1 && f <= kMaxKSplit && f <= sb) {
            g.ksplit = f;
            g.full = f > 1 ? 0 : tiles;
            return g;
        }
    }
    const int tail = tiles % sm_count;
    if (tail == 0)
        return g;
    const int full = tiles - tail;
    const double us_per_sb = 3.7, partial_bytes_per_us = 5.0e6, tile_bytes = double(tok) * kRows * 4;
    double best_t = 1e30;
    for (int ks = 1; ks <= kMaxKSplit && ks <= sb; ++ks) {
        const double waves = double((int64_t(tail) * ks + sm_count - 1) / sm_count);
        double t = waves * ((sb + ks - 1) / ks) * us_per_sb;
        if (ks > 1)
            t += double(ks) * tail * tile_bytes * 2.0 / partial_bytes_per_us;
        if (t < best_t - 1e-9) {
            best_t = t;
            g.ksplit = ks;
        }
    }
    g.full = g.ksplit > 1 ? full : tiles;
    return g;
}

size_t gemm_q4k_ws_floats(int64_t M, int64_t Ntot, int ksplit)
{
    // Partials keep Y's layout (the group's matrices side by side); only the
    // tail tiles' regions are written.
    return ksplit > 1 ? size_t(ksplit) * size_t(M) * size_t(Ntot) : 0;
}

cudaError_t launch_gemm_q4k(const GemmArgs &a, int sm_count, cudaStream_t s)
{
    GemmParams P;
    memset(&P, 0, sizeof(P));
    memcpy(&P.tm_x, a.tmap_x, sizeof(CUtensorMap));
    P.nmat = a.nmat;
    int rt = 0, off = 0;
    bool vec = true;
    for (int i = 0; i < a.nmat; ++i) {
        memcpy(&P.tm_hdr[i], a.tmap_hdr[i], sizeof(CUtensorMap));
        memcpy(&P.tm_nib[i], a.tmap_nib[i], sizeof(CUtensorMap));
        P.y[i] = a.y[i];
        P.n_rows[i] = int(a.N[i]);
        rt += int((a.N[i] + kRows - 1) / kRows);
        P.rt_end[i] = rt;
        P.col_off[i] = off;
        off += int(a.N[i]);
        vec = vec && a.N[i] % 4 == 0 && (reinterpret_cast<uintptr_t>(a.y[i]) & 15) == 0;
    }
    for (int i = a.nmat; i < kGemmMaxGroup; ++i)
        P.rt_end[i] = rt;
    P.Ntot = off;
    P.ws = a.ws;
    P.M = int(a.M);
    P.K = int(a.K);
    P.tok_tiles = int((a.M + a.tok - 1) / a.tok);
    P.tiles = P.tok_tiles * rt;
    P.ksplit = a.ksplit;
    P.full_units = a.ksplit > 1 ? a.full_tiles : P.tiles;
    P.units = P.full_units + (P.tiles - P.full_units) * P.ksplit;
    P.vec_store = vec ? 1 : 0;
    P.status = a.status;
    // Bulk-store epilogue: every Y_i (and the partials) as a tensor of fp32
    // rows, 32 x 32 boxes with the 128-byte swizzle of the staging buffers.
    bool tma = vec && getenv("QMM_GEMM_THREAD_STORES") == nullptr;
    for (int i = 0; i < a.nmat && tma; ++i)
        tma = encode_tmap_2d(&P.tm_y[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.y[i], uint64_t(a.N[i]),
                             uint64_t(a.M), uint64_t(a.N[i]) * 4, 32u, 32u,
                             CU_TENSOR_MAP_SWIZZLE_128B) == 0;
    if (tma && a.ksplit > 1)
        tma = encode_tmap_3d(&P.tm_ws, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.ws, uint64_t(P.Ntot),
                             uint64_t(a.M), uint64_t(a.ksplit), uint64_t(P.Ntot) * 4,
                             uint64_t(a.M) * uint64_t(P.Ntot) * 4, 32u, 32u, 1u,
                             CU_TENSOR_MAP_SWIZZLE_128B) == 0;
    P.tma_store = tma ? 1 : 0;
    const GemmInstance gi = pick_gemm(a.tok, a.fmt);
    const auto kern = gi.fn;
    const size_t smem = gi.smem;
    cudaError_t e = func_smem(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess)
        return e;
    int grid = sm_count < P.units ? sm_count : P.units;
    if (const char *g = getenv("QMM_GEMM_CTAS"))
        if (atoi(g) > 0 && atoi(g) < grid)
            grid = atoi(g);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    e = counted(cudaLaunchKernelEx(&cfg, kern, P));
    if (e != cudaSuccess || P.ksplit == 1)
        return e;
    ReduceParams R;
    memset(&R, 0, sizeof(R));
    for (int i = 0; i < kGemmMaxGroup; ++i) {
        R.y[i] = P.y[i];
        R.n_rows[i] = P.n_rows[i];
        R.col_off[i] = P.col_off[i];
        R.rt_end[i] = P.rt_end[i];
    }
    R.nmat = a.nmat;
    R.Ntot = P.Ntot;
    R.M = P.M;
    R.ks = P.ksplit;
    R.tok = a.tok;
    R.tok_tiles = P.tok_tiles;
    R.first_tail = P.full_units;
    R.n_tail = P.tiles - P.full_units;
    R.ws = a.ws;
    R.vec = vec ? 1 : 0;
    const int64_t work = int64_t(R.n_tail) * a.tok * (kRows / 4);
    int64_t blocks = (work + 255) / 256;
    if (blocks > int64_t(sm_count) * 16)
        blocks = int64_t(sm_count) * 16;
    cudaLaunchConfig_t rc = cfg;
    rc.gridDim = dim3(unsigned(blocks));
    rc.blockDim = dim3(256);
    rc.dynamicSmemBytes = 0;
    return counted(cudaLaunchKernelEx(&rc, splitk_reduce_kernel, R));
}

} // namespace qmm
