// moe_q8.cu -- the expert GEMV of moe.cu for Q8_0 weights.
//
// The operation is moe.cu's ("Frink Inference: the Rust alternative to
// llama.cpp", "Architecture coverage: 100 models with evidence"; Q8_0 is one
// of the formats of "Where llama.cpp is still ahead"), on the same bucketing:
// for a group of at most kGroupTokens slots of expert e, Y[slot, rows] =
// W_e x_slot, with gate and up optionally in one launch and SwiGLU applied
// there.
//
// Arithmetic, fp32 on the CUDA cores: a Q8_0 block is d (fp16) and 32 int8
// codes q; q becomes the float 2^23 + 128 + q with one byte permute (the
// code's byte, sign bit flipped, under the exponent byte 0x4B) and one
// packed subtraction, both exact; products accumulate per block in packed
// FFMA2 over (weight i, weight i+1) pairs, and the block sum is scaled by d
// once.  With the routing weight on the input (Llama 4) the slot's sum is
// multiplied by r afterwards: the same value as W (r x) up to rounding.
//
// Work.  An item is (group, row tile): 64 rows of one matrix, or 32 rows of
// gate and the same 32 rows of up.  An item's rows stream through shared
// memory one K-slice of 256 weights at a time: a stage holds the rows'
// 272-byte slices (two TMA boxes of 32 rows; rows 272 bytes apart, so the
// lanes of a quarter warp reading neighbouring rows hit disjoint banks) and
// the group's activations for the slice (one 1 KB bulk copy per token).  A
// producer warp fills a ring of stages; eight consumer warps take, in every
// stage, Q8_0 block w of the slice for warp w (weights 32w .. 32w+31) and
// rows l and l+32 for lane l, so a lane keeps its sums over the whole K in
// registers and the activations of a half block (16 weights x the group's
// tokens) serve both of its rows.  At the end of an item the eight warps'
// sums meet in shared memory and are added in warp order (bitwise
// repeatable), then stored (with silu(gate) * up when fused).  CTA b takes
// items b, b + G, b + 2G, ... of the (group, tile) sequence.
#include <cstring>

#include <cuda.h>
#include <cuda_fp16.h>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {

namespace {

constexpr int kQ8eWarps = 8;                   // consumer warps (one per block of a slice)
constexpr int kQ8eThreads = 32 * (kQ8eWarps + 1);
constexpr int kQ8eRows = 64;                   // rows per item (stage)
constexpr int kQ8eBoxRows = 32;                // rows per TMA box
constexpr int kQ8eSliceBytes = 272;            // 8 blocks of 34 bytes = 256 weights
constexpr int kQ8eWBytes = kQ8eRows * kQ8eSliceBytes;        // 17408
constexpr int kQ8eXBytes = kGroupTokens * 256 * 4;           // 4096
constexpr int kQ8eHdrBytes = 128;                            // item header (first stage)
constexpr int kQ8eStageBytes = kQ8eWBytes + kQ8eXBytes + kQ8eHdrBytes;  // 21632
constexpr int kQ8eRedFloats = kQ8eWarps * kQ8eRows * 4;      // one item's per-warp sums

static_assert(kGroupTokens == 4, "the consumer keeps four token sums per row");
static_assert(kQ8eStageBytes % 128 == 0, "stages start on 128-byte boundaries");

struct MoeQ8Params {
    CUtensorMap tmap[2];    // u32 view of the stacked experts' rows, box (68, 32)
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

__device__ __forceinline__ uint4 lds128(const void *p)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}

__device__ __forceinline__ float4 lds128f(const void *p)
{
    const uint4 v = lds128(p);
    return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                       __uint_as_float(v.w));
}

__device__ __forceinline__ void consumers_sync()
{
    asm volatile("bar.sync 1, %0;" ::"r"(32 * kQ8eWarps) : "memory");
}

// Words k = 0..3 of the 16 bytes starting I words (+ 2 bytes when sel is
// 0x5432) into the 32 bytes a ++ b.
template <int I>
__device__ __forceinline__ void pick4(const uint32_t (&a)[8], unsigned sel, uint32_t (&q)[4])
{
#pragma unroll
    for (int k = 0; k < 4; ++k)
        q[k] = __byte_perm(a[I + k], a[I + k + 1], sel);
}

// One row's half block: 16 codes (four words) against the half block's
// activations xv[t][0..15]; returns d * sum per token.
template <int NT>
__device__ __forceinline__ void half_block(const uint32_t (&q)[4], const float (&xv)[kGroupTokens][16],
                                           float d, float (&out)[kGroupTokens])
{
    const float2 off = make_float2(-8388736.f, -8388736.f);  // -(2^23 + 128)
    float2 acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t)
        acc[t] = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t u = q[k] ^ 0x80808080u;  // int8 -> 128 + q as a byte
        const float2 w01 = __fadd2_rn(make_float2(byte_magic(u, 0), byte_magic(u, 1)), off);
        const float2 w23 = __fadd2_rn(make_float2(byte_magic(u, 2), byte_magic(u, 3)), off);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            acc[t] = __ffma2_rn(w01, make_float2(xv[t][4 * k], xv[t][4 * k + 1]), acc[t]);
            acc[t] = __ffma2_rn(w23, make_float2(xv[t][4 * k + 2], xv[t][4 * k + 3]), acc[t]);
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t)
        out[t] = d * (acc[t].x + acc[t].y);
}

// One stage for one consumer lane: block w of the slice, rows l and l + 32.
template <int NT>
__device__ __forceinline__ void stage_dot(const uint8_t *st, int w, int lane,
                                          float (&run)[2][kGroupTokens])
{
    const float *xs = reinterpret_cast<const float *>(st + kQ8eWBytes);  // [4][256]
    const int blk = 34 * w;
    float d[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const uint8_t *row = st + (lane + 32 * r) * kQ8eSliceBytes;
        const uint32_t dw = *reinterpret_cast<const uint32_t *>(row + (blk & ~3));
        d[r] = __half2float(__ushort_as_half((unsigned short)((blk & 2) ? (dw >> 16) : (dw & 0xffffu))));
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        // the half block's activations (the same address in every lane)
        float xv[kGroupTokens][16];
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 v = lds128f(xs + t * 256 + 32 * w + 16 * h + 4 * k);
                xv[t][4 * k] = v.x;
                xv[t][4 * k + 1] = v.y;
                xv[t][4 * k + 2] = v.z;
                xv[t][4 * k + 3] = v.w;
            }
        // codes 16h .. 16h+15 of the block start at byte o of the row slice
        const int o = blk + 2 + 16 * h;
        const int a16 = o & ~15;
        const unsigned sel = (o & 2) ? 0x5432u : 0x3210u;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const uint8_t *row = st + (lane + 32 * r) * kQ8eSliceBytes;
            const uint4 A = lds128(row + a16), B = lds128(row + a16 + 16);
            const uint32_t a[8] = {A.x, A.y, A.z, A.w, B.x, B.y, B.z, B.w};
            uint32_t q[4];
            switch ((o >> 2) & 3) {
            case 0: pick4<0>(a, sel, q); break;
            case 1: pick4<1>(a, sel, q); break;
            case 2: pick4<2>(a, sel, q); break;
            default: pick4<3>(a, sel, q); break;
            }
            float s[kGroupTokens];
            half_block<NT>(q, xv, d[r], s);
#pragma unroll
            for (int t = 0; t < NT; ++t)
                run[r][t] += s[t];
        }
    }
}

__global__ void __launch_bounds__(kQ8eThreads, 1) moe_q8_kernel(const __grid_constant__ MoeQ8Params P)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int NS = P.nstage;
    uint8_t *stages = smem;
    float *red = reinterpret_cast<float *>(smem + size_t(NS) * kQ8eStageBytes);  // [2][8][64][4]
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
                for (int j = 0; j < P.NB; ++j, ++k) {
                    const int slot = int(k % NS);
                    if (k >= NS &&
                        !mbar_wait_bounded(&empty[slot], unsigned((k / NS - 1) & 1))) {
                        atomicOr(P.status, kStatusTimeoutBit);
                        s_fail = 1;
                        failed = true;
                        break;
                    }
                    uint8_t *st = stages + size_t(slot) * kQ8eStageBytes;
                    if (j == 0) {  // the item's token count and slots
                        int *hdr = reinterpret_cast<int *>(st + kQ8eWBytes + kQ8eXBytes);
                        hdr[0] = grp.z;
#pragma unroll
                        for (int m = 0; m < kGroupTokens; ++m)
                            hdr[1 + m] = sA[m];
                    }
                    mbar_arrive_expect_tx(&full[slot], unsigned(kQ8eWBytes + grp.z * 1024));
                    if (P.nmat == 2) {
                        tma_box(st, &P.tmap[0], j * 68, y0, &full[slot], pw);
                        tma_box(st + kQ8eBoxRows * kQ8eSliceBytes, &P.tmap[1], j * 68, y0,
                                &full[slot], pw);
                    } else {
                        tma_box(st, &P.tmap[0], j * 68, y0, &full[slot], pw);
                        tma_box(st + kQ8eBoxRows * kQ8eSliceBytes, &P.tmap[0], j * 68,
                                y0 + kQ8eBoxRows, &full[slot], pw);
                    }
#pragma unroll
                    for (int m = 0; m < kGroupTokens; ++m)
                        if (m < grp.z) {
                            const int64_t xrow = P.x_per_slot ? sA[m] : sA[m] / P.top_k;
                            bulk_g2s(st + kQ8eWBytes + m * 1024, P.x + xrow * P.ldx + j * 256,
                                     1024u, &full[slot], px);
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
    // the (row, token) this thread stores at the end of an item
    const int t_mine = P.nmat == 2 ? (i < kQ8eBoxRows * kGroupTokens ? i / kQ8eBoxRows : -1)
                                   : i / kQ8eRows;
    const int r_mine = P.nmat == 2 ? (i & (kQ8eBoxRows - 1)) : (i & (kQ8eRows - 1));
    for (int64_t it = blockIdx.x; it < n_items; it += gridDim.x, ib ^= 1) {
        const int tt = int(it % P.tpm);
        int cnt = 0, s_mine = -1;
        float sc_mine = 1.f;
        float run[2][kGroupTokens];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int t = 0; t < kGroupTokens; ++t)
                run[r][t] = 0.f;
        for (int j = 0; j < P.NB; ++j, ++k) {
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
            const uint8_t *st = stages + size_t(slot) * kQ8eStageBytes;
            if (j == 0) {
                const int *hdr = reinterpret_cast<const int *>(st + kQ8eWBytes + kQ8eXBytes);
                cnt = hdr[0];
                s_mine = (t_mine >= 0 && t_mine < cnt) ? hdr[1 + t_mine] : -1;
                if (P.xscale && s_mine >= 0)
                    sc_mine = __ldg(P.xscale + s_mine);  // used at the end of the item
            }
            if (cnt <= 2)
                stage_dot<2>(st, warp, lane, run);
            else
                stage_dot<kGroupTokens>(st, warp, lane, run);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[slot]);
        }
        // the warps' sums of this item, then their sum in warp order
        float *rb = red + ib * kQ8eRedFloats;
#pragma unroll
        for (int r = 0; r < 2; ++r)
            *reinterpret_cast<float4 *>(rb + (warp * kQ8eRows + lane + 32 * r) * 4) =
                make_float4(run[r][0], run[r][1], run[r][2], run[r][3]);
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

size_t moe_q8_smem(int nstage)
{
    return size_t(nstage) * kQ8eStageBytes + size_t(2) * kQ8eRedFloats * sizeof(float) +
           size_t(2) * nstage * sizeof(uint64_t);
}

int moe_q8_stages() { return 8; }

int encode_moe_q8_map(void *out128, const void *w, int64_t N, int64_t row_bytes)
{
    return encode_tmap_2d(out128, CU_TENSOR_MAP_DATA_TYPE_UINT32, w, uint64_t(row_bytes / 4),
                          uint64_t(N), uint64_t(row_bytes), 68u, uint32_t(kQ8eBoxRows),
                          CU_TENSOR_MAP_SWIZZLE_NONE);
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
    P.nstage = moe_q8_stages();
    const size_t smem = moe_q8_smem(P.nstage);
    cudaError_t e = func_smem(reinterpret_cast<const void *>(moe_q8_kernel), smem);
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
    return counted(cudaLaunchKernelEx(&cfg, moe_q8_kernel, P));
}

} // namespace qmm
