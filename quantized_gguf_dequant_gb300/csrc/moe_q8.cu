// moe_q8.cu -- the expert GEMV of moe.cu for Q8_0 weights.
//
// The operation is moe.cu's ("Frink Inference: the Rust alternative to
// llama.cpp", "Architecture coverage: 100 models with evidence"; Q8_0 is one
// of the formats of "Where llama.cpp is still ahead"), on the same bucketing:
// for a group of at most kGroupTokens slots of expert e, Y[slot, rows] =
// W_e x_slot, with gate and up optionally in one launch and SwiGLU applied
// there.
//
// Arithmetic, on the tensor cores (mma.sync m16n8k16, fp16 operands, fp32
// accumulation): a Q8_0 block is d (fp16) and 32 int8 codes q.  Each code
// enters the MMA as u = q + 128 (one XOR flips the sign bits; one byte
// permute puts two codes into the low bytes of an fp16 pair, u * 2^-24, an
// exact subnormal).  The B columns are the group's four tokens, each as two
// fp16 terms (hi + lo) of its activations scaled by a power of two per block
// and token, so every product is exact and one MMA per 16 weights serves all
// four tokens.  Per block and token: sum q x = sum u x - 128 X (X the
// block's activation sum), times d, added in fp32.  With the routing weight
// on the input (Llama 4) the slot's sum is multiplied by r afterwards: the
// same value as W (r x) up to rounding.
//
// Work.  An item is (group, row tile): 64 rows of one matrix, or 32 rows of
// gate and the same 32 rows of up.  An item's rows stream through shared
// memory two K-slices of 256 weights at a time (one where a row has an odd
// number of slices): a stage holds the rows' 544-byte pieces (two TMA boxes
// of 32 rows over a u64 view of the rows) and the group's activations for
// those slices (one bulk copy per token).  Longer row pieces per stage
// measured faster than one slice (185 against 270 us per OLMoE layer).  A
// producer warp fills a ring of stages; eight consumer warps take, in every
// slice of a stage, Q8_0 block w for warp w (weights 32w .. 32w+31, two MMA
// k-steps) over all 64 rows (four 16-row MMA tiles), preparing the block's
// B fragments once; lane (g, c) keeps, over the whole K, the sums of rows g
// and g+8 of each tile for token c.  At the end of an item the eight warps'
// sums meet in shared memory and are added in warp order (bitwise
// repeatable), then stored (with silu(gate) * up when fused).  CTA b takes
// items b, b + G, b + 2G, ... of the (group, tile) sequence.
#include <cstring>

#include <cuda.h>
#include <cuda_fp16.h>

#include "qmm_device.cuh"
#include "qmm_internal.h"
#include "tc_common.cuh"

namespace qmm {

namespace {

constexpr int kQ8eWarps = 8;                   // consumer warps (one per block of a slice)
constexpr int kQ8eThreads = 32 * (kQ8eWarps + 1);
constexpr int kQ8eRows = 64;                   // rows per item (stage)
constexpr int kQ8eBoxRows = 32;                // rows per TMA box
constexpr int kQ8eHdrBytes = 128;              // item header (first stage)
constexpr int kQ8eRedFloats = kQ8eWarps * kQ8eRows * 4;      // one item's per-warp sums

// A stage holds SPS K-slices of 256 weights (SPS = 2 where the row has an
// even number of slices: 544-byte row pieces, half as many stages per item).
template <int SPS>
struct Q8eShape {
    static constexpr int kSlice = 272 * SPS;                   // bytes of a row in a stage
    static constexpr int kW = kQ8eRows * kSlice;               // weight bytes of a stage
    static constexpr int kX = kGroupTokens * 256 * SPS * 4;    // activations of a stage
    static constexpr int kStage = kW + kX + kQ8eHdrBytes;
    static constexpr int kStages = SPS == 1 ? 8 : 4;
    static_assert(kStage % 128 == 0, "stages start on 128-byte boundaries");
};

static_assert(kGroupTokens == 4, "the consumer keeps four token sums per row");

struct MoeQ8Params {
    CUtensorMap tmap[2];    // u64 view of the stacked experts' rows, box (34 * SPS, 32)
    float *y[2];
    const float *x;
    int64_t ldx;
    const int4 *groups;
    const int *slots;
    const int *n_groups;
    unsigned *status;
    const float *xscale;    // per-slot routing weight applied on the input, or null
    int Ne;                 // rows per expert
    int NB;                 // 256-weight slices per row
    int nmat;               // 1, or 2 (gate and up)
    int fuse;               // nmat == 2: y[0] = silu(gate) * up
    int tpm;                // row tiles per group
    int top_k;
    int x_per_slot;
    int nstage;
};

__device__ __forceinline__ float silu(float z) { return z / (1.f + expf(-z)); }

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void tma_box(void *dst, const CUtensorMap *map, int x, int y,
                                        uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void consumers_sync()
{
    asm volatile("bar.sync 1, %0;" ::"r"(32 * kQ8eWarps) : "memory");
}

__device__ __forceinline__ uint32_t lds32(const void *p)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)));
    return v;
}

__device__ __forceinline__ uint32_t lds_u16(const void *p)
{
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(smem_u32(p)));
    return v;
}

__device__ __forceinline__ uint32_t pack_half2(__half a, __half b)
{
    return uint32_t(__half_as_ushort(a)) | (uint32_t(__half_as_ushort(b)) << 16);
}

// One stage for one consumer lane (g, c) of warp w: block w of the slice over
// the stage's four 16-row tiles.  k-step h (0, 1) covers codes 16h .. 16h+15
// of the block; lane column c supplies codes 16h + 4c .. +3: (4c, 4c+1) in
// k-slots (2c, 2c+1), (4c+2, 4c+3) in (2c+8, 2c+9).  B column n is token n/2,
// term n%2 (hi, lo).  run[t][r]: row 16t + g + 8r, token c.
template <int SPS>
__device__ __forceinline__ void stage_mma(const uint8_t *st, int sl, int w, int lane, int cnt,
                                          float (&run)[4][2])
{
    using S = Q8eShape<SPS>;
    const int g = lane >> 2, c = lane & 3;
    const int tk = g >> 1, term = g & 1;  // the B column this lane supplies
    // slice sl of the stage: activations [4][256 * SPS] from + sl * 256, rows
    // S::kSlice bytes apart from + sl * 272
    const float *xs = reinterpret_cast<const float *>(st + S::kW) + sl * 256;
    const int xst = 256 * SPS;
    // ---- B: the block's activations of token tk, scaled by 2^s (s per block
    // and token: the largest |x| below 2^15), split into hi + lo halves
    float4 v[2];
#pragma unroll
    for (int h = 0; h < 2; ++h)
        v[h] = tk < cnt ? *reinterpret_cast<const float4 *>(xs + tk * xst + 32 * w + 16 * h + 4 * c)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
    uint32_t mb = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h)
        mb = max(mb, max(max(__float_as_uint(v[h].x) & 0x7fffffffu, __float_as_uint(v[h].y) & 0x7fffffffu),
                         max(__float_as_uint(v[h].z) & 0x7fffffffu, __float_as_uint(v[h].w) & 0x7fffffffu)));
    mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
    mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
    const int s = mb ? 14 - (int(mb >> 23) - 127) : 0;
    float xsum = (v[0].x + v[0].y) + (v[0].z + v[0].w) + ((v[1].x + v[1].y) + (v[1].z + v[1].w));
    xsum += __shfl_xor_sync(0xffffffffu, xsum, 1);
    xsum += __shfl_xor_sync(0xffffffffu, xsum, 2);
    uint32_t b[2][2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const float e[4] = {scale_pow2(v[h].x, s), scale_pow2(v[h].y, s), scale_pow2(v[h].z, s),
                            scale_pow2(v[h].w, s)};
        __half q[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half hi = __float2half_rn(e[i]);
            q[i] = term ? __float2half_rn(e[i] - __half2float(hi)) : hi;
        }
        b[h][0] = pack_half2(q[0], q[1]);
        b[h][1] = pack_half2(q[2], q[3]);
    }
    // the D side is token c: its scale and block sum from lane (2c, 0)
    const int sc_ = __shfl_sync(0xffffffffu, s, 8 * c);
    const float off = -128.f * __shfl_sync(0xffffffffu, xsum, 8 * c);
    // ---- A: four codes of rows g and g+8 of each tile per k-step
    const int blk = 34 * w;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint8_t *r0 = st + (16 * t + g) * S::kSlice + sl * 272;
        const uint8_t *r1 = r0 + 8 * S::kSlice;
        float d[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int o = blk + 2 + 16 * h + 4 * c;  // 4-byte aligned when w is odd
            uint32_t wa, wb;
            if (w & 1) {
                wa = lds32(r0 + o);
                wb = lds32(r1 + o);
            } else {
                wa = __byte_perm(lds32(r0 + o - 2), lds32(r0 + o + 2), 0x5432u);
                wb = __byte_perm(lds32(r1 + o - 2), lds32(r1 + o + 2), 0x5432u);
            }
            wa ^= 0x80808080u;  // u = q + 128
            wb ^= 0x80808080u;
            const uint32_t a0 = __byte_perm(wa, 0u, 0x4140u), a1 = __byte_perm(wb, 0u, 0x4140u);
            const uint32_t a2 = __byte_perm(wa, 0u, 0x4342u), a3 = __byte_perm(wb, 0u, 0x4342u);
            if (h == 0)
                tc::mma16816_zero(d, a0, a1, a2, a3, b[h][0], b[h][1]);
            else
                tc::mma16816(d, a0, a1, a2, a3, b[h][0], b[h][1]);
        }
        const float d0 = __half2float(__ushort_as_half((unsigned short)lds_u16(r0 + blk)));
        const float d1 = __half2float(__ushort_as_half((unsigned short)lds_u16(r1 + blk)));
        // sum u x = (hi + lo columns) * 2^24 * 2^-s (two exact power-of-two steps)
        const float u0 = scale_pow2((d[0] + d[1]) * 16777216.f, -sc_);
        const float u1 = scale_pow2((d[2] + d[3]) * 16777216.f, -sc_);
        run[t][0] = fmaf(d0, u0 + off, run[t][0]);
        run[t][1] = fmaf(d1, u1 + off, run[t][1]);
    }
}

template <int SPS>
__global__ void __launch_bounds__(kQ8eThreads, 1) moe_q8_kernel(const __grid_constant__ MoeQ8Params P)
{
    using S = Q8eShape<SPS>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int NS = P.nstage;
    const int NJ = P.NB / SPS;  // stages per item
    uint8_t *stages = smem;
    float *red = reinterpret_cast<float *>(smem + size_t(NS) * S::kStage);  // [2][8][64][4]
    uint64_t *full = reinterpret_cast<uint64_t *>(red + 2 * kQ8eRedFloats);
    uint64_t *empty = full + NS;
    __shared__ int s_fail;

    const int warp = int(threadIdx.x) >> 5, lane = int(threadIdx.x) & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kQ8eWarps);
        }
        fence_barrier_init();
        s_fail = 0;
    }
    __syncthreads();
    pdl_wait();  // the bucket tables, x and y belong to earlier kernels until here
    pdl_launch_dependents();

    const int64_t n_items = int64_t(*P.n_groups) * P.tpm;
    const int rows_per_mat = P.nmat == 2 ? kQ8eBoxRows : kQ8eRows;

    if (warp == kQ8eWarps) {
        // ---------------- producer (lane 0)
        if (lane == 0) {
            const uint64_t pw = policy_evict_first(), px = policy_evict_last();
            int64_t k = 0;
            bool failed = false;
            const int64_t G = gridDim.x;
            // The group record of an item is fetched two items ahead and its
            // slots one item ahead, so the issue of stages never waits on them.
            const int4 none = make_int4(0, 0, 0, 0);
            int64_t it = blockIdx.x;
            int4 gA = it < n_items ? P.groups[it / P.tpm] : none;
            int4 gB = it + G < n_items ? P.groups[(it + G) / P.tpm] : none;
            int sA[kGroupTokens];
#pragma unroll
            for (int m = 0; m < kGroupTokens; ++m)
                sA[m] = m < gA.z ? P.slots[gA.y + m] : -1;
            for (; it < n_items && !failed; it += G) {
                int sB[kGroupTokens];
#pragma unroll
                for (int m = 0; m < kGroupTokens; ++m)
                    sB[m] = m < gB.z ? P.slots[gB.y + m] : -1;
                const int4 gC = it + 2 * G < n_items ? P.groups[(it + 2 * G) / P.tpm] : none;
                const int tt = int(it % P.tpm);
                const int4 grp = gA;
                const int y0 = grp.x * P.Ne + tt * rows_per_mat;
                for (int j = 0; j < NJ; ++j, ++k) {
                    const int slot = int(k % NS);
                    if (k >= NS &&
                        !mbar_wait_bounded(&empty[slot], unsigned((k / NS - 1) & 1))) {
                        atomicOr(P.status, kStatusTimeoutBit);
                        s_fail = 1;
                        failed = true;
                        break;
                    }
                    uint8_t *st = stages + size_t(slot) * S::kStage;
                    if (j == 0) {  // the item's token count and slots
                        int *hdr = reinterpret_cast<int *>(st + S::kW + S::kX);
                        hdr[0] = grp.z;
#pragma unroll
                        for (int m = 0; m < kGroupTokens; ++m)
                            hdr[1 + m] = sA[m];
                    }
                    mbar_arrive_expect_tx(&full[slot], unsigned(S::kW + grp.z * 1024 * SPS));
                    const int xw = j * 34 * SPS;  // u64 words into the row
                    if (P.nmat == 2) {
                        tma_box(st, &P.tmap[0], xw, y0, &full[slot], pw);
                        tma_box(st + kQ8eBoxRows * S::kSlice, &P.tmap[1], xw, y0, &full[slot], pw);
                    } else {
                        tma_box(st, &P.tmap[0], xw, y0, &full[slot], pw);
                        tma_box(st + kQ8eBoxRows * S::kSlice, &P.tmap[0], xw, y0 + kQ8eBoxRows,
                                &full[slot], pw);
                    }
#pragma unroll
                    for (int m = 0; m < kGroupTokens; ++m)
                        if (m < grp.z) {
                            const int64_t xrow = P.x_per_slot ? sA[m] : sA[m] / P.top_k;
                            bulk_g2s(st + S::kW + m * 1024 * SPS, P.x + xrow * P.ldx + j * 256 * SPS,
                                     1024u * SPS, &full[slot], px);
                        }
                }
                gA = gB;
                gB = gC;
#pragma unroll
                for (int m = 0; m < kGroupTokens; ++m)
                    sA[m] = sB[m];
            }
            if (failed) {
                // Let the copies in flight land before shared memory is released.
                const int64_t k0 = k > NS ? k - NS : 0;
                for (int64_t kk = k0; kk < k; ++kk)
                    mbar_wait_bounded(&full[kk % NS], unsigned((kk / NS) & 1), 100000000ll);
            }
        }
        return;
    }

    // ---------------- consumers
    int64_t k = 0;
    int ib = 0;  // item parity: which half of red[]
    const int i = int(threadIdx.x);  // 0 .. 255
    // the (row, token) this thread stores at the end of an item (if any)
    const int t_mine = P.nmat == 2 ? (i < kQ8eBoxRows * kGroupTokens ? i / kQ8eBoxRows : -1)
                                   : (i < kQ8eRows * kGroupTokens ? i / kQ8eRows : -1);
    const int r_mine = P.nmat == 2 ? (i & (kQ8eBoxRows - 1)) : (i & (kQ8eRows - 1));
    for (int64_t it = blockIdx.x; it < n_items; it += gridDim.x, ib ^= 1) {
        const int tt = int(it % P.tpm);
        int cnt = 0, s_mine = -1;
        float sc_mine = 1.f;
        float run[4][2];
#pragma unroll
        for (int t = 0; t < 4; ++t)
            run[t][0] = run[t][1] = 0.f;
        for (int j = 0; j < NJ; ++j, ++k) {
            const int slot = int(k % NS);
            if (*reinterpret_cast<volatile int *>(&s_fail))
                break;
            if (!mbar_wait_bounded(&full[slot], unsigned((k / NS) & 1))) {
                if (lane == 0) {
                    atomicOr(P.status, kStatusTimeoutBit);
                    s_fail = 1;
                }
                break;
            }
            const uint8_t *st = stages + size_t(slot) * S::kStage;
            if (j == 0) {
                const int *hdr = reinterpret_cast<const int *>(st + S::kW + S::kX);
                cnt = hdr[0];
                s_mine = (t_mine >= 0 && t_mine < cnt) ? hdr[1 + t_mine] : -1;
                if (P.xscale && s_mine >= 0)
                    sc_mine = __ldg(P.xscale + s_mine);  // used at the end of the item
            }
#pragma unroll
            for (int sl = 0; sl < SPS; ++sl)
                stage_mma<SPS>(st, sl, warp, lane, cnt, run);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[slot]);
        }
        // the warps' sums of this item, then their sum in warp order
        float *rb = red + ib * kQ8eRedFloats;
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int r = 0; r < 2; ++r)
                rb[(warp * kQ8eRows + 16 * t + (lane >> 2) + 8 * r) * 4 + (lane & 3)] = run[t][r];
        consumers_sync();
        if (*reinterpret_cast<volatile int *>(&s_fail))
            break;
        auto total = [&](int row, int t) {
            float s = 0.f;
            for (int w = 0; w < kQ8eWarps; ++w)
                s += rb[(w * kQ8eRows + row) * 4 + t];
            return s;
        };
        const int s = s_mine;
        if (P.nmat == 2) {
            const int row = tt * kQ8eBoxRows + r_mine;
            if (s >= 0 && row < P.Ne) {
                const float g = sc_mine * total(r_mine, t_mine);
                const float u = sc_mine * total(kQ8eBoxRows + r_mine, t_mine);
                if (P.fuse) {
                    P.y[0][int64_t(s) * P.Ne + row] = silu(g) * u;
                } else {
                    P.y[0][int64_t(s) * P.Ne + row] = g;
                    P.y[1][int64_t(s) * P.Ne + row] = u;
                }
            }
        } else {
            const int row = tt * kQ8eRows + r_mine;
            if (s >= 0 && row < P.Ne)
                P.y[0][int64_t(s) * P.Ne + row] = sc_mine * total(r_mine, t_mine);
        }
    }
}

} // namespace

// Slices per stage for rows of NB 256-weight slices.
// (Four slices per stage measured slower: two stages in flight and 4-way
// bank conflicts at a 1088-byte row stride.)
int moe_q8_sps(int64_t NB) { return NB % 2 == 0 ? 2 : 1; }

size_t moe_q8_smem(int sps)
{
    const size_t stage = sps == 2 ? size_t(Q8eShape<2>::kStage) : size_t(Q8eShape<1>::kStage);
    const int ns = sps == 2 ? Q8eShape<2>::kStages : Q8eShape<1>::kStages;
    return size_t(ns) * stage + size_t(2) * kQ8eRedFloats * sizeof(float) +
           size_t(2) * ns * sizeof(uint64_t);
}

int encode_moe_q8_map(void *out128, const void *w, int64_t N, int64_t row_bytes)
{
    const int sps = moe_q8_sps(row_bytes / 272);
    return encode_tmap_2d(out128, CU_TENSOR_MAP_DATA_TYPE_UINT64, w, uint64_t(row_bytes / 8),
                          uint64_t(N), uint64_t(row_bytes), uint32_t(34 * sps),
                          uint32_t(kQ8eBoxRows), CU_TENSOR_MAP_SWIZZLE_NONE);
}

cudaError_t launch_moe_q8(const MoeExpertArgs &a, int sm_count, cudaStream_t s)
{
    MoeQ8Params P;
    memset(&P, 0, sizeof(P));
    for (int i = 0; i < a.nmat; ++i) {
        memcpy(&P.tmap[i], a.tmap[i], sizeof(CUtensorMap));
        P.y[i] = a.y[i];
    }
    P.x = a.x;
    P.ldx = a.ldx;
    P.groups = a.ix.groups;
    P.slots = a.ix.slots;
    P.n_groups = a.ix.n_groups;
    P.status = a.status;
    P.xscale = a.xscale;
    P.Ne = int(a.Ne);
    P.NB = int(a.K / 256);
    P.nmat = a.nmat;
    P.fuse = a.fuse_swiglu;
    const int rows = a.nmat == 2 ? kQ8eBoxRows : kQ8eRows;
    P.tpm = int((a.Ne + rows - 1) / rows);
    P.top_k = a.top_k;
    P.x_per_slot = a.x_per_slot;
    const int sps = moe_q8_sps(P.NB);
    P.nstage = sps == 2 ? Q8eShape<2>::kStages : Q8eShape<1>::kStages;
    const size_t smem = moe_q8_smem(sps);
    const auto kern = sps == 2 ? moe_q8_kernel<2> : moe_q8_kernel<1>;
    cudaError_t e = func_smem(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(sm_count));
    cfg.blockDim = dim3(kQ8eThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return counted(cudaLaunchKernelEx(&cfg, kern, P));
}

} // namespace qmm
