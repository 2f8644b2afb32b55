// gemv.cu -- decode GEMV y = W x with the GGUF blocks decoded in registers
// (Q4_K and Q8_0), the weights streamed through shared memory by the TMA
// engine, a deterministic split-K, and programmatic dependent launch.
//
// The operation: "Building a Rust Inference Engine That Matches Llama.cpp",
// "Where the wins came from" -- quantized weights never become a
// full-precision buffer; the dequant math happens inline in the dot product.
//
// Work decomposition.  A CTA owns a contiguous range of rows (ranges are
// balanced to within one row) and one K-slice.  Its threads form row teams;
// thread c of a team owns the 64-weight chunk c of the slice for the whole
// kernel: its 64 activations are loaded once, pre-scaled, and kept in
// registers while the team walks the rows.  Rows arrive in shared memory in
// stages (a ring of `stages` buffers, one bulk copy per contiguous run of
// rows, completion tracked by an mbarrier transaction count).  Each thread
// reads its chunk's bytes of a row from shared memory, decodes and
// multiplies, and the team's partial sums meet in a shuffle tree and a
// fixed-order sum over the team's warps.  With split-K the K-slices' partial
// rows go to the workspace and the last CTA of a row range (atomic ticket)
// adds them in slice order, so results are bitwise repeatable.
//
// Q4_K decode without integer-to-float conversions.  For a nibble q sitting
// at bit p (p <= 20) of a 32-bit word, masking the word leaves the bit
// pattern q * 2^p, and a bit pattern v < 2^24 read as a float is exactly
// v * 2^-149 (a subnormal, or the smallest normal binade, whose spacing is
// the same).  So float(word & (15 << p)) = q * 2^(p-149) exactly, with one
// LOP3.  Each activation is pre-scaled by 2^(149-p-E) for the bit position p
// of the nibble it meets (E chosen per chunk from its largest |x| so that
// nothing overflows), and one packed fp32 FMA (FFMA2, Blackwell) multiplies
// the low and the high nibble of a byte -- sub-blocks 2c and 2c+1 -- by their
// activations at once.  Per sub-block the sum S is then scaled back:
// contribution = d*sc*S*2^E - dmin*m*X, X the plain sum of the sub-block's
// activations.
#include <cstdio>
#include <cstdlib>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {

namespace {

constexpr int kMaxThreads = 256;
constexpr int kStageBytesTarget = 18432;
constexpr int kStages = 4;

struct __align__(16) U4 {
    uint32_t a, b, c, d;
};

__device__ __forceinline__ U4 lds128(const uint8_t *p)
{
    return *reinterpret_cast<const U4 *>(p);
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    return __ffma2_rn(a, b, c);
}

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

// Where a global row lives: matrix index and row within it.
__device__ __forceinline__ int matrix_of(const GemvArgs &a, int64_t row)
{
    int m = 0;
#pragma unroll
    for (int i = 0; i < kMaxGroup - 1; ++i)
        if (i < a.nmat - 1 && row >= a.row_end[i])
            m = i + 1;
    return m;
}

__device__ __forceinline__ int64_t row_start(const GemvArgs &a, int m)
{
    return m == 0 ? 0 : a.row_end[m - 1];
}

// ----------------------------------------------------------------- per-thread
// decode state (activations of the owned chunk, in registers).

struct Q4State {
    float xl[32], xh[32];  // pre-scaled activations for low / high nibbles
    float Xl, Xh;          // plain sums of the two sub-block halves
    float p1, p2;          // 2^E = p1 * p2
    uint32_t selA, selB, mA, mB, mC, mD;
    int hdr_off, qs_off;   // byte offsets of the chunk's header and quants in a row
};

__device__ __forceinline__ void q4_prologue(Q4State &st, const float *x, int64_t gchunk,
                                            int local_chunk)
{
    const int64_t blk = gchunk >> 2;
    const int c4 = int(gchunk & 3);
    const float4 *xv = reinterpret_cast<const float4 *>(x + blk * 256 + c4 * 64);
    float raw_l[32], raw_h[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float4 a = __ldg(xv + i);
        float4 b = __ldg(xv + 8 + i);
        raw_l[4 * i + 0] = a.x; raw_l[4 * i + 1] = a.y; raw_l[4 * i + 2] = a.z; raw_l[4 * i + 3] = a.w;
        raw_h[4 * i + 0] = b.x; raw_h[4 * i + 1] = b.y; raw_h[4 * i + 2] = b.z; raw_h[4 * i + 3] = b.w;
    }
    uint32_t mbits = 0;
    float sl = 0.f, sh = 0.f;
#pragma unroll
    for (int l = 0; l < 32; ++l) {
        mbits = max(mbits, __float_as_uint(raw_l[l]) & 0x7fffffffu);
        mbits = max(mbits, __float_as_uint(raw_h[l]) & 0x7fffffffu);
        sl += raw_l[l];
        sh += raw_h[l];
    }
    // Largest |x| < 2^(eM+1); E = eM + 23 keeps every pre-scaled activation
    // below 2^127 and puts the largest product near 2^-19.
    const int eM = int(mbits >> 23) - 127;
    const int E = eM + 23;
#pragma unroll
    for (int l = 0; l < 32; ++l) {
        const int i = l & 3;
        const int p_lo = (i < 3) ? 8 * i : 0;  // byte 3 is shifted down by 24 first
        st.xl[l] = scale_pow2(raw_l[l], 149 - p_lo - E);
        st.xh[l] = scale_pow2(raw_h[l], 149 - (p_lo + 4) - E);
    }
    st.Xl = sl;
    st.Xh = sh;
    const int E1 = E / 2;
    st.p1 = exp2i(E1);
    st.p2 = exp2i(E - E1);
    // Scale/min bytes of sub-blocks 2c4, 2c4+1 (see the Q4_K packing).
    const uint32_t u0 = 2u * uint32_t(c4 & 1);
    st.selA = u0 | ((u0 + 1) << 4) | ((4 + u0) << 8) | ((5 + u0) << 12);
    st.selB = u0 | ((u0 + 1) << 4) | (u0 << 8) | ((u0 + 1) << 12);
    if (c4 < 2) {
        st.mA = 0x3F3F3F3Fu; st.mB = 0; st.mC = 0; st.mD = 0;
    } else {
        st.mA = 0; st.mB = 0x30303030u; st.mC = 0x00000F0Fu; st.mD = 0x0F0F0000u;
    }
    st.hdr_off = (local_chunk >> 2) * 144;
    st.qs_off = st.hdr_off + 16 + 32 * c4;
}

// Partial dot product of one row's chunk (64 weights) with the chunk's
// activations, in natural units.
__device__ __forceinline__ float q4_row(const Q4State &st, const uint8_t *row)
{
    const U4 h = lds128(row + st.hdr_off);
    const U4 q0 = lds128(row + st.qs_off);
    const U4 q1 = lds128(row + st.qs_off + 16);
    const uint32_t qw[8] = {q0.a, q0.b, q0.c, q0.d, q1.a, q1.b, q1.c, q1.d};
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t w = qw[t];
        const uint32_t w3 = w >> 24;
        float2 &acc = (t & 1) ? acc1 : acc0;
        acc = ffma2(make_float2(as_float(w & 0x0000000Fu), as_float(w & 0x000000F0u)),
                    make_float2(st.xl[4 * t + 0], st.xh[4 * t + 0]), acc);
        acc = ffma2(make_float2(as_float(w & 0x00000F00u), as_float(w & 0x0000F000u)),
                    make_float2(st.xl[4 * t + 1], st.xh[4 * t + 1]), acc);
        acc = ffma2(make_float2(as_float(w & 0x000F0000u), as_float(w & 0x00F00000u)),
                    make_float2(st.xl[4 * t + 2], st.xh[4 * t + 2]), acc);
        acc = ffma2(make_float2(as_float(w3 & 0x0Fu), as_float(w3 & 0xF0u)),
                    make_float2(st.xl[4 * t + 3], st.xh[4 * t + 3]), acc);
    }
    const float2 S = __fadd2_rn(acc0, acc1);
    // (sc_lo, sc_hi, m_lo, m_hi) as bytes of R.
    const uint32_t A = __byte_perm(h.b, h.c, st.selA);
    const uint32_t B = __byte_perm(h.d, h.d, st.selB);
    const uint32_t R = (A & st.mA) | ((A >> 2) & st.mB) | (B & st.mC) | ((B >> 4) & st.mD);
    const float2 magic = make_float2(-8388608.f, -8388608.f);
    const float2 sc = __fadd2_rn(make_float2(byte_magic(R, 0), byte_magic(R, 1)), magic);
    const float2 mm = __fadd2_rn(make_float2(byte_magic(R, 2), byte_magic(R, 3)), magic);
    const float2 us = __fmul2_rn(sc, S);
    const float u = us.x + us.y;
    const float v = fmaf(mm.x, st.Xl, mm.y * st.Xh);
    const float2 dd = half2_bits_to_float2(h.a);  // (d, dmin)
    const float t = (dd.x * u) * st.p1;
    return fmaf(t, st.p2, -(dd.y * v));
}

struct Q8State {
    float xa[32], xb[32];  // activations of the chunk's two blocks
    int off;               // byte offset of the chunk in a row
};

__device__ __forceinline__ void q8_prologue(Q8State &st, const float *x, int64_t gchunk,
                                            int local_chunk)
{
    const float4 *xv = reinterpret_cast<const float4 *>(x + gchunk * 64);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float4 a = __ldg(xv + i);
        float4 b = __ldg(xv + 8 + i);
        st.xa[4 * i + 0] = a.x; st.xa[4 * i + 1] = a.y; st.xa[4 * i + 2] = a.z; st.xa[4 * i + 3] = a.w;
        st.xb[4 * i + 0] = b.x; st.xb[4 * i + 1] = b.y; st.xb[4 * i + 2] = b.z; st.xb[4 * i + 3] = b.w;
    }
    st.off = local_chunk * 68;
}

// Two Q8_0 blocks (68 bytes, 4-byte aligned): block A = bytes 0..33, block B
// = bytes 34..67.  int8 q -> float exactly: flip the sign bit (q + 128 as an
// unsigned byte), drop the byte into the mantissa of 2^23 and subtract
// 2^23 + 128.
__device__ __forceinline__ float q8_row(const Q8State &st, const uint8_t *row)
{
    const uint32_t *p = reinterpret_cast<const uint32_t *>(row + st.off);
    uint32_t w[17];
#pragma unroll
    for (int i = 0; i < 17; ++i)
        w[i] = p[i];
    const float2 d = half2_bits_to_float2(__byte_perm(w[0], w[8], 0x7610));
    const float2 off = make_float2(-8388736.f, -8388736.f);  // -(2^23 + 128)
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t qa = __funnelshift_r(w[k], w[k + 1], 16) ^ 0x80808080u;
        const uint32_t qb = w[9 + k] ^ 0x80808080u;
        float2 &acc = (k & 1) ? acc1 : acc0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 q = __fadd2_rn(make_float2(byte_magic(qa, i), byte_magic(qb, i)), off);
            acc = ffma2(q, make_float2(st.xa[4 * k + i], st.xb[4 * k + i]), acc);
        }
    }
    const float2 S = __fadd2_rn(acc0, acc1);
    return fmaf(d.x, S.x, d.y * S.y);
}

// ----------------------------------------------------------------- kernel
struct KParams {
    GemvArgs a;
    int kchunks, team, rg, rpg, stage_rows, stages, ksplit, row_slices;
    int64_t slice_bytes;
};

template <int FMT>
__global__ void __launch_bounds__(kMaxThreads, 2) gemv_kernel(const __grid_constant__ KParams P)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const GemvArgs &a = P.a;
    const int tid = threadIdx.x;
    const int rs = blockIdx.x / P.ksplit;  // row slice
    const int ks = blockIdx.x % P.ksplit;  // K-slice
    // Balanced contiguous row range of this slice.
    const int64_t base = a.N / P.row_slices, extra = a.N % P.row_slices;
    const int64_t r0 = rs * base + min64(rs, extra);
    const int64_t r1 = r0 + base + (rs < extra ? 1 : 0);
    const int64_t nrows = r1 - r0;
    const int nst = int((nrows + P.stage_rows - 1) / P.stage_rows);

    const size_t stage_bytes = size_t(P.stage_rows) * size_t(P.slice_bytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + size_t(P.stages) * stage_bytes);
    const int nwt = (P.team + 31) / 32;  // warps per team
    float *red = reinterpret_cast<float *>(full + P.stages);  // [2][stage_rows][nwt]
    int *flag = reinterpret_cast<int *>(red + 2 * P.stage_rows * nwt);

    uint64_t policy = 0;
    if (tid == 0) {
        for (int s = 0; s < P.stages; ++s)
            mbar_init(&full[s], 1);
        fence_barrier_init();
        *flag = 0;
        policy = policy_evict_first();
    }
    __syncthreads();
    pdl_launch_dependents();

    // Producer: stage s -> buffer s % stages.  The weights are constant, so
    // the first stages are requested before waiting for the previous kernel.
    auto issue = [&](int s) {
        const int64_t ra = r0 + int64_t(s) * P.stage_rows;
        const int64_t rb = min64(ra + P.stage_rows, r1);
        uint8_t *dst = smem + size_t(s % P.stages) * stage_bytes;
        uint64_t *bar = &full[s % P.stages];
        mbar_arrive_expect_tx(bar, unsigned((rb - ra) * P.slice_bytes));
        if (P.ksplit == 1) {
            int64_t r = ra;
            while (r < rb) {
                const int m = matrix_of(a, r);
                const int64_t seg_end = min64(rb, a.row_end[m]);
                const uint8_t *src = a.w[m] + (r - row_start(a, m)) * a.row_bytes;
                bulk_g2s(dst + (r - ra) * P.slice_bytes, src, unsigned((seg_end - r) * a.row_bytes),
                         bar, policy);
                r = seg_end;
            }
        } else {
            for (int64_t r = ra; r < rb; ++r) {
                const int m = matrix_of(a, r);
                const uint8_t *src =
                    a.w[m] + (r - row_start(a, m)) * a.row_bytes + int64_t(ks) * P.slice_bytes;
                bulk_g2s(dst + (r - ra) * P.slice_bytes, src, unsigned(P.slice_bytes), bar, policy);
            }
        }
    };
    int issued = 0;
    if (tid == 0) {
        for (; issued < min(P.stages, nst); ++issued)
            issue(issued);
    }

    pdl_wait();  // x (and y / workspace) belong to the previous kernel until here

    const int g = tid / P.team;         // row team
    const int c = tid % P.team;         // chunk lane within the team
    const bool active = (g < P.rg) && (c < P.kchunks);
    const int64_t gchunk = int64_t(ks) * P.kchunks + c;

    Q4State s4;
    Q8State s8;
    if (active) {
        if (FMT == QMM_Q4_K)
            q4_prologue(s4, a.x, gchunk, c);
        else
            q8_prologue(s8, a.x, gchunk, c);
    }
    const int lane = tid & 31;
    const int width = P.team < 32 ? P.team : 32;
    const int warp_in_team = c >> 5;

    bool failed = false;
    for (int s = 0; s < nst; ++s) {
        const int buf = s % P.stages;
        if (!mbar_wait_bounded(&full[buf], unsigned(s / P.stages) & 1u)) {
            atomicOr(a.status, kStatusTimeoutBit);
            *flag = 1;
        }
        const uint8_t *stage = smem + size_t(buf) * stage_bytes;
        const int64_t ra = r0 + int64_t(s) * P.stage_rows;
        const int nr = int(min64(P.stage_rows, r1 - ra));
        float *rd = red + (s & 1) * P.stage_rows * nwt;
#pragma unroll 1
        for (int j = 0; j < P.rpg; ++j) {
            const int i = g + P.rg * j;  // row within the stage
            float part = 0.f;
            if (active && i < nr && !*flag) {
                const uint8_t *row = stage + size_t(i) * P.slice_bytes;
                part = (FMT == QMM_Q4_K) ? q4_row(s4, row) : q8_row(s8, row);
            }
            part = warp_sum(part, width);
            if ((c & 31) == 0 && g < P.rg && i < nr)
                rd[i * nwt + warp_in_team] = part;
        }
        __syncthreads();  // stage buffer free; partial sums visible
        if (*flag) {
            failed = true;
            break;
        }
        if (tid < nr) {
            float v = 0.f;
            for (int wv = 0; wv < nwt; ++wv)
                v += rd[tid * nwt + wv];
            const int64_t row = ra + tid;
            if (P.ksplit == 1) {
                const int m = matrix_of(a, row);
                a.y[m][row - row_start(a, m)] = v;
            } else {
                a.ws[int64_t(ks) * a.N + row] = v;
            }
        }
        if (tid == 0 && issued < nst) {
            fence_proxy_async_smem();
            issue(issued++);
        }
    }

    if (failed) {
        // Let the copies still in flight land before the CTA's shared memory
        // is released (bounded as well).
        if (tid == 0) {
            for (int s = 0; s < issued; ++s)
                mbar_wait_bounded(&full[s % P.stages], unsigned(s / P.stages) & 1u, 100000000ll);
        }
        return;
    }

    if (P.ksplit > 1) {
        __shared__ int last;
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            const unsigned old = atomicAdd(&a.tickets[rs], 1u);
            last = (old == unsigned(P.ksplit - 1));
        }
        __syncthreads();
        if (last) {
            __threadfence();
            for (int64_t r = r0 + tid; r < r1; r += blockDim.x) {
                float v = 0.f;
                for (int k = 0; k < P.ksplit; ++k)
                    v += __ldcg(a.ws + int64_t(k) * a.N + r);
                const int m = matrix_of(a, r);
                a.y[m][r - row_start(a, m)] = v;
            }
            if (tid == 0)
                a.tickets[rs] = 0u;
        }
    }
}

} // namespace

GemvPlan plan_gemv(int fmt, int64_t N, int64_t K, int sm_count, int force_ksplit)
{
    GemvPlan p;
    const int64_t chunks = K / 64;  // K % 256 == 0 for both formats here
    // K-slices: at most 256 chunks each (one thread per chunk), whole Q4_K
    // blocks (a multiple of 4 chunks), and enough CTAs to cover the GPU when
    // there are few rows.
    // A valid split cuts the row into equal slices of whole 256-weight blocks.
    const int64_t nblocks = chunks / 4;
    auto valid = [&](int64_t ks) { return ks >= 1 && ks <= nblocks && nblocks % ks == 0; };
    int ksplit = int((chunks + kMaxThreads - 1) / kMaxThreads);
    while (!valid(ksplit))
        ++ksplit;
    const int64_t target_ctas = int64_t(sm_count) * 2;
    while (force_ksplit <= 0 && N * ksplit < target_ctas && valid(int64_t(ksplit) * 2))
        ksplit *= 2;
    if (force_ksplit > 0 && valid(force_ksplit) && chunks / force_ksplit <= kMaxThreads)
        ksplit = force_ksplit;
    p.ksplit = ksplit;
    p.kchunks = int(chunks / ksplit);
    int team = 1;
    if (p.kchunks <= 32) {
        while (team < p.kchunks)
            team *= 2;
    } else {
        team = (p.kchunks + 31) / 32 * 32;
    }
    p.rg = kMaxThreads / team;
    if (p.rg < 1)
        p.rg = 1;
    p.threads = p.rg * team;
    p.slice_bytes = (fmt == QMM_Q4_K) ? int64_t(p.kchunks / 4) * 144 : int64_t(p.kchunks) * 68;
    int rpg = int(kStageBytesTarget / (int64_t(p.rg) * p.slice_bytes));
    rpg = rpg < 1 ? 1 : (rpg > 4 ? 4 : rpg);
    p.rpg = rpg;
    p.stage_rows = p.rg * rpg;
    p.stages = kStages;
    int64_t slices = target_ctas / ksplit;
    if (slices > N)
        slices = N;
    if (slices < 1)
        slices = 1;
    p.row_slices = int(slices);
    const int nwt = (team + 31) / 32;
    p.smem = size_t(p.stages) * size_t(p.stage_rows) * size_t(p.slice_bytes) +
             size_t(p.stages) * 8 + size_t(2 * p.stage_rows * nwt) * 4 + 16;
    return p;
}

size_t gemv_workspace_floats(const GemvPlan &p, int64_t N)
{
    return p.ksplit > 1 ? size_t(p.ksplit) * size_t(N) : 0;
}

static int team_of(const GemvPlan &p) { return p.threads / p.rg; }

cudaError_t launch_gemv(const GemvPlan &p, const GemvArgs &a, cudaStream_t s)
{
    KParams P;
    P.a = a;
    P.kchunks = p.kchunks;
    P.team = team_of(p);
    P.rg = p.rg;
    P.rpg = p.rpg;
    P.stage_rows = p.stage_rows;
    P.stages = p.stages;
    P.ksplit = p.ksplit;
    P.row_slices = p.row_slices;
    P.slice_bytes = p.slice_bytes;

    void (*kern)(KParams) = (a.fmt == QMM_Q4_K) ? gemv_kernel<QMM_Q4_K> : gemv_kernel<QMM_Q8_0>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(p.smem));
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(p.row_slices * p.ksplit));
    cfg.blockDim = dim3(unsigned(p.threads));
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, P);
}

} // namespace qmm
