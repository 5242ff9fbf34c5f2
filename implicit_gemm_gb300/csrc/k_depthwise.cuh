// Depthwise (C = K = 1 per group) weight gradient on CUDA cores.
//
//     dW[g, tap] = sum over pixels p of dY[p, g] * X[p shifted by tap, g]
//
// A depthwise group makes both implicit-GEMM operands single channels, so the
// per-group GEMM is 1 x YX x N*Ho*Wo: no dense contraction is left for the
// tensor cores.  Following the group-merge idea of PR #12359 ("add group
// merging (Gm) for depthwise grouped conv"), Gm adjacent groups are handled
// together so that the channel run -- contiguous in NHWGC / NHWGK -- becomes
// the vector axis: each thread owns Gm consecutive channels (a 2*Gm-byte
// vector) and all YX taps of them.  Merging divides the parallelism by Gm and
// the pixel split (the "split-K" of this kernel) multiplies it back.
//
// A CTA owns CB channels and a slice of (n, row-strip) tiles.  A producer warp
// streams each tile's X rows (with halo, zero-filled outside the image by TMA)
// and dY rows into a shared-memory ring; compute threads (channel vector,
// output row, column segment) accumulate in registers, then reduce over the
// CTA through shared memory and over splits via atomics or the workspace.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace wg {

struct DwParams {
    int G, Ho, Wo, Y, X, T;
    int sh, sw, dh, dw, plh, plw;
    int CB, R, nseg, seg_len, nused;
    int xw, xh, n_hstrips, per_split, total_tiles;
    int stages, x_bytes_al, stage_bytes, x_tx, dy_tx;
    int mode, out_dtype;
    void* out;
    WsLayout ws;  // split-K workspace layout (mode 3)
};


// The arithmetic works on the 16-bit inputs as loaded: a packed register holds
// two channels, and the mixed-precision FMA (fp32 accumulator, bf16 or fp16
// factors) multiplies them without converting first.  The product of two
// 16-bit floats is exact in fp32, so the result equals fmaf on the converted
// values bit for bit.
template <bool BF16>
__device__ __forceinline__ void fma2(float& a0, float& a1, uint32_t x, uint32_t y)
{
    if constexpr (BF16)
        asm("{\n\t.reg .b16 xl, xh, yl, yh;\n\tmov.b32 {xl, xh}, %2;\n\tmov.b32 {yl, yh}, %3;\n\t"
            "fma.rn.f32.bf16 %0, xl, yl, %0;\n\tfma.rn.f32.bf16 %1, xh, yh, %1;\n\t}"
            : "+f"(a0), "+f"(a1)
            : "r"(x), "r"(y));
    else
        asm("{\n\t.reg .b16 xl, xh, yl, yh;\n\tmov.b32 {xl, xh}, %2;\n\tmov.b32 {yl, yh}, %3;\n\t"
            "fma.rn.f32.f16 %0, xl, yl, %0;\n\tfma.rn.f32.f16 %1, xh, yh, %1;\n\t}"
            : "+f"(a0), "+f"(a1)
            : "r"(x), "r"(y));
}

template <bool BF16>
__device__ __forceinline__ void fma1(float& a0, uint32_t x, uint32_t y)
{
    if constexpr (BF16)
        asm("{\n\t.reg .b16 xl, xh, yl, yh;\n\tmov.b32 {xl, xh}, %1;\n\tmov.b32 {yl, yh}, %2;\n\t"
            "fma.rn.f32.bf16 %0, xl, yl, %0;\n\t}"
            : "+f"(a0)
            : "r"(x), "r"(y));
    else
        asm("{\n\t.reg .b16 xl, xh, yl, yh;\n\tmov.b32 {xl, xh}, %1;\n\tmov.b32 {yl, yh}, %2;\n\t"
            "fma.rn.f32.f16 %0, xl, yl, %0;\n\t}"
            : "+f"(a0)
            : "r"(x), "r"(y));
}

// A vector of GM channels as packed pairs (GM = 1: the low half of one word).
template <int GM>
struct Packed {
    static constexpr int N = GM >= 2 ? GM / 2 : 1;
    uint32_t w[N];
};

template <int GM>
__device__ __forceinline__ void load_vec(const uint16_t* p, Packed<GM>& v)
{
    if constexpr (GM == 8) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        v.w[0] = u.x, v.w[1] = u.y, v.w[2] = u.z, v.w[3] = u.w;
    } else if constexpr (GM == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        v.w[0] = u.x, v.w[1] = u.y;
    } else if constexpr (GM == 2) {
        v.w[0] = *reinterpret_cast<const uint32_t*>(p);
    } else {
        v.w[0] = *p;
    }
}

// acc[t][j] += x[j] * dy[j] over the vector's channels.
template <bool BF16, int GM>
__device__ __forceinline__ void fma_vec(float (&acc)[GM], const Packed<GM>& x, const Packed<GM>& dy)
{
    if constexpr (GM == 1) {
        fma1<BF16>(acc[0], x.w[0], dy.w[0]);
    } else {
#pragma unroll
        for (int q = 0; q < GM / 2; ++q) fma2<BF16>(acc[2 * q], acc[2 * q + 1], x.w[q], dy.w[q]);
    }
}

// One window column: the X vectors of the three filter rows at one input column.
template <int GM>
__device__ __forceinline__ void load_col3(const uint16_t* r0, const uint16_t* r1, const uint16_t* r2, int off,
                                          Packed<GM> (&w)[3])
{
    load_vec<GM>(r0 + off, w[0]);
    load_vec<GM>(r1 + off, w[1]);
    load_vec<GM>(r2 + off, w[2]);
}

// acc[y*3 + x] += dY(pixel) * X(row y, column x of the window (c0, c1, c2)).
template <bool BF16, int GM>
__device__ __forceinline__ void fma_col3(const uint16_t* dyp, const Packed<GM> (&c0)[3], const Packed<GM> (&c1)[3],
                                         const Packed<GM> (&c2)[3], float (&acc)[9][GM])
{
    Packed<GM> dy;
    load_vec<GM>(dyp, dy);
#pragma unroll
    for (int y = 0; y < 3; ++y) {
        fma_vec<BF16, GM>(acc[y * 3 + 0], c0[y], dy);
        fma_vec<BF16, GM>(acc[y * 3 + 1], c1[y], dy);
        fma_vec<BF16, GM>(acc[y * 3 + 2], c2[y], dy);
    }
}

// Vectors of 8 channels hold 72 accumulators plus a 36-register window of
// packed pairs: one CTA per SM.  Narrower vectors fit two CTAs per SM.
template <bool BF16, int GM, bool SLIDE3>
__global__ void __launch_bounds__(288, GM >= 8 ? 1 : 2)
    depthwise_wgrad_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmy,
                           const __grid_constant__ DwParams p)
{
    constexpr int MAXT = 9;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_shared<uint8_t>(smem_raw, 1024);
    const int nthreads = blockDim.x - 32;
    const int red_bytes = nthreads * p.T * GM * 4;
    uint8_t* tail = smem + max(p.stages * p.stage_bytes, red_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(tail);
    uint64_t* empty = full + 8;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cb = blockIdx.x, split = blockIdx.y;
    const int t0 = split * p.per_split;
    const int ntl = max(0, min(p.per_split, p.total_tiles - t0));
    const int n_cwarps = nthreads >> 5;

    // The kernel launched after this one (the split reduction, or the next
    // call's first kernel) may be scheduled at once; it waits for this whole
    // grid's results before it reads them.
    pdl_launch_dependents();
    // Row tile i of this split into ring stage i % stages: X rows with halo, dY rows.
    auto issue_tile = [&](int i) {
        const int st = i % p.stages;
        const int tile = t0 + i;
        const int n = tile / p.n_hstrips;
        const int ho0 = (tile - n * p.n_hstrips) * p.R;
        uint8_t* sb = smem + st * p.stage_bytes;
        mbar_arrive_expect_tx(&full[st], (uint32_t)(p.x_tx + p.dy_tx));
        tma_load_5d(sb, &tmx, &full[st], cb * p.CB, -p.plw, ho0 * p.sh - p.plh, 0, n);
        tma_load_5d(sb + p.x_bytes_al, &tmy, &full[st], cb * p.CB, 0, ho0, 0, n);
    };
    // Thread 0 initialises the barriers and issues the first tile before the
    // block barrier, so that the TMA unit's first fetch of the tensor maps
    // overlaps the prologue; the producer warp continues from the second tile.
    const int pre = ntl > 0 ? 1 : 0;
    if (tid == 0) {
        if (pre) {
            tma_prefetch_desc(&tmx);
            tma_prefetch_desc(&tmy);
        }
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], (uint32_t)n_cwarps);
        }
        fence_mbar_init();
        // A programmatic dependent of the kernel before it on the stream: unless
        // that is this call's zeroing kernel (which waited for everything before
        // it), X and dY are read only after it has finished.
        if (p.mode != 2) pdl_wait();
        for (int i = 0; i < pre; ++i) issue_tile(i);
    }
    __syncthreads();

    float acc[MAXT][GM];
#pragma unroll
    for (int t = 0; t < MAXT; ++t)
#pragma unroll
        for (int j = 0; j < GM; ++j) acc[t][j] = 0.f;

    const int NV = p.CB / GM;
    const int CB = p.CB, Wo = p.Wo, xw = p.xw, sh = p.sh, dh = p.dh;
    if (warp == n_cwarps) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            for (int i = pre; i < ntl; ++i) {
                const int st = i % p.stages;
                const uint32_t ph = (uint32_t)(i / p.stages) & 1u;
                if (i >= p.stages && !mbar_wait(&empty[st], ph ^ 1u)) break;
                issue_tile(i);
            }
        }
    } else {
        // ------------------------------------------------ compute threads
        const int v = tid % NV, rest = tid / NV;
        const int seg = rest % p.nseg, r = rest / p.nseg;
        const int wo_a = seg * p.seg_len, wo_b = min(p.Wo, wo_a + p.seg_len);
        const bool active = tid < p.nused && wo_a < wo_b;
        // Per-tile work is kept small: the thread's offsets inside a stage are
        // the same for every tile, and the tile's row strip advances by one
        // (the tiles of a split are consecutive) instead of being divided out.
        const int cv = v * GM;
        const int x_off = (r * sh) * xw * CB + cv, y_off = (r * Wo) * CB + cv;
        // General filters: each tap's offset from the pixel's first X vector.
        int tap_off[MAXT];
#pragma unroll
        for (int t = 0; t < MAXT; ++t) {
            const int tt = t < p.T ? t : 0;
            const int ty = tt / p.X, tx = tt - (tt / p.X) * p.X;
            tap_off[t] = (ty * p.dh * p.xw + tx * p.dw) * p.CB;
        }
        int strip = t0 % p.n_hstrips;
        int st = 0;
        uint32_t ph = 0;
        for (int i = 0; i < ntl; ++i) {
            if (!mbar_wait(&full[st], ph)) break;
            const int ho0 = strip * p.R;
            strip = strip + 1 == p.n_hstrips ? 0 : strip + 1;
            if (active && ho0 + r < p.Ho) {
                const uint16_t* xs = reinterpret_cast<const uint16_t*>(smem + st * p.stage_bytes);
                const uint16_t* ys = reinterpret_cast<const uint16_t*>(smem + st * p.stage_bytes + p.x_bytes_al);
                if constexpr (SLIDE3) {
                    // 3x3 filter, stride 1 and dilation 1 along W: a 3x3 window of
                    // X vectors slides along the row, one new column per pixel.
                    // Unrolled by 3 so the three window columns change roles
                    // instead of being copied.
                    const int CBv = CB;
                    const uint16_t* xr0 = xs + x_off;
                    const uint16_t* xr1 = xr0 + dh * xw * CBv;
                    const uint16_t* xr2 = xr1 + dh * xw * CBv;
                    const uint16_t* yr = ys + y_off;
                    Packed<GM> wa[3], wb[3], wc[3];
                    load_col3<GM>(xr0, xr1, xr2, wo_a * CBv, wa);
                    load_col3<GM>(xr0, xr1, xr2, (wo_a + 1) * CBv, wb);
                    int wo = wo_a;
                    for (; wo + 3 <= wo_b; wo += 3) {
                        load_col3<GM>(xr0, xr1, xr2, (wo + 2) * CBv, wc);
                        fma_col3<BF16, GM>(yr + wo * CBv, wa, wb, wc, acc);
                        load_col3<GM>(xr0, xr1, xr2, (wo + 3) * CBv, wa);
                        fma_col3<BF16, GM>(yr + (wo + 1) * CBv, wb, wc, wa, acc);
                        load_col3<GM>(xr0, xr1, xr2, (wo + 4) * CBv, wb);
                        fma_col3<BF16, GM>(yr + (wo + 2) * CBv, wc, wa, wb, acc);
                    }
                    if (wo < wo_b) {
                        load_col3<GM>(xr0, xr1, xr2, (wo + 2) * CBv, wc);
                        fma_col3<BF16, GM>(yr + wo * CBv, wa, wb, wc, acc);
                        if (wo + 1 < wo_b) {
                            load_col3<GM>(xr0, xr1, xr2, (wo + 3) * CBv, wa);
                            fma_col3<BF16, GM>(yr + (wo + 1) * CBv, wb, wc, wa, acc);
                        }
                    }
                } else {
                    for (int wo = wo_a; wo < wo_b; ++wo) {
                        Packed<GM> dy;
                        load_vec<GM>(ys + y_off + wo * CB, dy);
                        const uint16_t* xb = xs + x_off + wo * p.sw * CB;
#pragma unroll
                        for (int t = 0; t < MAXT; ++t) {
                            if (t < p.T) {
                                Packed<GM> xv;
                                load_vec<GM>(xb + tap_off[t], xv);
                                fma_vec<BF16, GM>(acc[t], xv, dy);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            if (++st == p.stages) st = 0, ph ^= 1u;
        }
    }
    __syncthreads();
    // ---------------------------------------------------- reduce over the CTA
    // Thread tid holds channel vector v = tid % NV of slot tid / NV (a row and
    // column segment of the tile).  When NV divides 32, each warp first adds its
    // 32 / NV slots with a butterfly of shuffles (lanes l and l ^ m, m = 16, 8,
    // ... down to NV; the steps are unrolled so that the 9 * GM chains
    // interleave), lanes 0..NV-1 store the warp's sums, and the warps' sums are
    // added in warp order.  Otherwise every slot is stored and the slots are
    // added in order.  Both orders are fixed: the result is reproducible.
    float* red = reinterpret_cast<float*>(smem);
    const bool shfl = NV < 32 && (32 % NV) == 0;
    int nparts;
    if (shfl) {
        nparts = n_cwarps;
        if (warp < n_cwarps) {
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) {
                if (m < NV) break;
#pragma unroll
                for (int t = 0; t < MAXT; ++t)
#pragma unroll
                    for (int j = 0; j < GM; ++j) acc[t][j] += __shfl_xor_sync(0xffffffffu, acc[t][j], m);
            }
            if (lane < NV) {
#pragma unroll
                for (int t = 0; t < MAXT; ++t)
                    if (t < p.T)
#pragma unroll
                        for (int j = 0; j < GM; ++j) red[(warp * p.CB + lane * GM + j) * p.T + t] = acc[t][j];
            }
        }
    } else {
        nparts = p.nused / NV;
        if (tid < p.nused) {
            const int slot = tid / NV, v = tid % NV;
#pragma unroll
            for (int t = 0; t < MAXT; ++t)
                if (t < p.T)
#pragma unroll
                    for (int j = 0; j < GM; ++j) red[(slot * p.CB + v * GM + j) * p.T + t] = acc[t][j];
        }
    }
    __syncthreads();
    // One output (c, t) per thread, idx = c * T + t (the parts are stored in
    // that order, so that the reads are consecutive words): the parts added in
    // order.  dW index o = g * T + t; its workspace offset uses 32-bit
    // arithmetic (the depthwise workspace is one row of G * T < 2^31 elements).
    const int TC = p.T * p.CB, W = p.ws.W;
    // Atomic accumulation: wait for the kernel that zeroes dW (see
    // zero_f32_kernel); in the other modes this returns at once.  Every thread
    // passes it before its first global write.
    pdl_wait();
    for (int idx = tid; idx < TC; idx += blockDim.x) {
        const int c = idx / p.T, t = idx - c * p.T;
        float s = 0.f;
        for (int sl = 0; sl < nparts; ++sl) s += red[sl * TC + idx];
        const int g = cb * p.CB + c;
        if (g >= p.G) continue;
        const int o = g * p.T + t;
        if (p.mode == 2) {
            if (ntl > 0) red_add_f32(static_cast<float*>(p.out) + o, s);
        } else if (p.mode == 3) {
            const int jw = o / W;
            static_cast<float*>(p.out)[((long long)jw * p.ws.S + split) * W + (o - jw * W)] = s;
        } else if (p.out_dtype == 2) {
            static_cast<float*>(p.out)[o] = s;
        } else if (p.out_dtype == 0) {
            static_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(s);
        } else {
            static_cast<__half*>(p.out)[o] = __float2half_rn(s);
        }
    }
}

}  // namespace wg
