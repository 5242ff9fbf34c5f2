// Backward-data (dgrad) of the grouped convolution on the tensor cores:
//
//   dX[n, i, g, c] = sum over k and taps t with (i + pl - t*dil) / stride integral
//                    of dY[n, (i + pl - t*dil) / stride, g, k] * W[g, k, t, c]
//
// with dY positions outside the output reading zero (the adjoint of the forward
// convolution in X).  Strides split each dim's input positions into phases
// i = r + stride * j; within a phase the contributing taps read dY at j plus a
// fixed offset, so each phase is a stride-1 problem over its own tap list
// (tables in DgParams::dim, built on the host).  The pages' dgrad keeps dY (NHWGK) M-outer, its reduction
// axis k already contiguous, and reads W as KYXC; here the GEMM is
// D[pixel, c] += dY[pixel, k] * W[k, c] per tap, with:
//
//  * M = 128 input pixels of one image and depth slice: an 8 (w) x 16 (h) box,
//    or 128 along w for 1-D problems, in the MMA's sixteen 8-row groups;
//  * A = a dY halo patch in shared memory (rows = dY pixels, 128 bytes = 64 k
//    channels, K-major, 128-byte swizzle).  Every tap reads the same patch from
//    a row offset -- the descriptor start moves by whole rows, the 8-row groups
//    are a patch row apart -- so dY is loaded once per (K chunk, filter plane),
//    not once per tap;
//  * B = W tiles (rows = k, 128 bytes = 64 c, MN-major), one per tap, loaded
//    from a (C, taps, K, G) view of W so that k beyond the group reads zero;
//  * fp32 accumulators in TMEM; all eight warps store dX (one pixel per lane).
//
// Warp roles as in the weight-gradient kernel: warp 0 lane 0 issues TMA into
// an mbarrier ring, warp 1 issues the MMAs, every wait is bounded.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "plan.h"
#include "ptx.cuh"

namespace wg {

struct DgParams {
    int G, C, K, X, Y;  // groups, channels as the kernel sees them (folded: G blocks of C and K)
    int ch_pix;         // channels of one dX pixel (all groups)
    int ch_lim;         // channel bound of a block's stores (the real G*C)
    int Wi, Hi, Di;     // dX extents
    int bw, bh, PW, PH;
    int Nt, n_catoms, n_kc, TG;
    int n_tw, n_th, n_td;
    int patch_bytes, stage_bytes, stages, tmem_cols;
    uint32_t idesc;
    int out_dtype;  // wg_dtype of dX
    void* out;
    DgDim dim[3];   // stride phases along (w, h, d): positions, dY offsets, taps and their row shifts
};

constexpr int kDgThreads = 256;
constexpr int kDgMaxStages = 4;
constexpr uint32_t kDgWTile = 8192;  // one W tile: 64 k rows x 64 c

// Store 8 consecutive channels of one pixel (16 bytes of bf16/fp16, 32 of fp32).
__device__ __forceinline__ void store8(void* out, long long i, const float* v, int out_dtype)
{
    if (out_dtype == 2) {
        float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + i);
        o[0] = make_float4(v[0], v[1], v[2], v[3]);
        o[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else if (out_dtype == 0) {
        uint4 u;
        uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
            w[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + i) = u;
    } else {
        uint4 u;
        uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __half2 h = __floats2half2_rn(v[2 * j], v[2 * j + 1]);
            w[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(static_cast<__half*>(out) + i) = u;
    }
}

// n (16 or 32) consecutive TMEM columns of this warp's lanes, one wait.
__device__ __forceinline__ void dg_ld(uint32_t taddr, int n, float (&v)[32])
{
    uint32_t r[32];
    tmem_ld16_issue(taddr, r);
    if (n > 16) tmem_ld16_issue(taddr + 16u, r + 16);
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    reg_fence16(r);
    if (n > 16) reg_fence16(r + 16);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = i < 16 || n > 16 ? __uint_as_float(r[i]) : 0.f;
}

// Block-diagonal copy of W for a group fold of Gm: for block b,
//   We[b][k'][t][c'] = W[b*Gm + k'/K][k' % K][t][c' % C] where k'/K == c'/C and
//                      that group exists, else 0
// (16-bit words copied as they are).
__global__ void __launch_bounds__(256)
    dgrad_fold_w_kernel(const uint16_t* __restrict__ w, uint16_t* __restrict__ we, int G, int K, int C, int T, int Gm,
                        long long n)
{
    const int Km = Gm * K, Cm = Gm * C;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        long long r = i;
        const int cp = (int)(r % Cm);
        r /= Cm;
        const int t = (int)(r % T);
        r /= T;
        const int kp = (int)(r % Km);
        const long long b = r / Km;
        const int gl = kp / K;
        const long long g = b * Gm + gl;
        uint16_t v = 0;
        if (cp / C == gl && g < G) v = w[((g * K + kp % K) * T + t) * C + cp % C];
        we[i] = v;
    }
}

__global__ void __launch_bounds__(kDgThreads, 1)
    dgrad_kernel(const __grid_constant__ CUtensorMap tmy, const __grid_constant__ CUtensorMap tmw,
                 const __grid_constant__ DgParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_shared<uint8_t>(smem_raw, 1024);
    uint8_t* tail = smem + p.stages * p.stage_bytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(tail);
    uint64_t* empty = full + kDgMaxStages;
    uint64_t* accb = empty + kDgMaxStages;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(accb + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Tile: stride phase (pw, ph, pd), box (tw, th) of phase positions, depth
    // position td and image n.
    long long t = blockIdx.x;
    const DgDim& DW = p.dim[0];
    const DgDim& DH = p.dim[1];
    const DgDim& DD = p.dim[2];
    const int pw = (int)(t % DW.nph);
    t /= DW.nph;
    const int ph = (int)(t % DH.nph);
    t /= DH.nph;
    const int pd = (int)(t % DD.nph);
    t /= DD.nph;
    const int tw = (int)(t % p.n_tw);
    t /= p.n_tw;
    const int th = (int)(t % p.n_th);
    t /= p.n_th;
    const int td = (int)(t % p.n_td);
    const int n = (int)(t / p.n_td);
    const int ct = blockIdx.y, g = blockIdx.z;
    const int j0w = tw * p.bw, j0h = th * p.bh, c0 = ct * p.Nt;
    const int nx = DW.ntap[pw], ny = DH.ntap[ph], nz = DD.ntap[pd];
    const int nyx = nx * ny, TG = p.TG;
    const int n_tg = (nyx + TG - 1) / TG;
    // A tile with no position in its phase, or a phase no tap reaches, does no MMAs.
    const bool any = j0w < DW.J[pw] && j0h < DH.J[ph] && td < DD.J[pd];
    const int nk = any ? p.n_kc * nz * n_tg : 0;
    const int stages = p.stages, stage_bytes = p.stage_bytes, patch_bytes = p.patch_bytes;
    const int n_catoms = p.n_catoms, X = p.X;

    if (threadIdx.x == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(accb, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 1) {
        tmem_alloc(tslot, (uint32_t)p.tmem_cols);
        tmem_relinquish();
        tc_fence_before();
    }
    uint32_t tbase = 0;
    if (warp != 0) {
        named_bar_sync(1, kDgThreads - 32);  // warps 1..7: the allocation is done
        tc_fence_after();
        tbase = *tslot;
    }

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            tma_prefetch_desc(&tmy);
            tma_prefetch_desc(&tmw);
            const uint32_t patch_tx = (uint32_t)(p.PW * p.PH * 128);
            for (int i = 0; i < nk; ++i) {
                const int st = i % stages;
                const uint32_t ph2 = (uint32_t)(i / stages) & 1u;
                if (i >= stages && !mbar_wait(&empty[st], ph2 ^ 1u)) break;
                const int tg = i % n_tg, rest = i / n_tg;
                const int zi = rest % nz, kc = rest / nz;
                const int y0 = tg * TG, ntap = min(TG, nyx - y0);
                const int z = DD.tap[pd][zi];
                uint8_t* sb = smem + st * stage_bytes;
                mbar_arrive_expect_tx(&full[st], patch_tx + (uint32_t)(ntap * n_catoms) * kDgWTile);
                // The dY rows the box's positions read for every (y, x) tap of plane z.
                tma_load_5d(sb, &tmy, &full[st], g * p.K + kc * 64, j0w + DW.qmin[pw], j0h + DH.qmin[ph],
                            td + DD.qmin[pd] + DD.shift[pd][zi], n);
                for (int j = 0; j < ntap; ++j) {
                    const int yi = (y0 + j) / nx, xi = (y0 + j) - yi * nx;
                    const int tap = (z * p.Y + DH.tap[ph][yi]) * X + DW.tap[pw][xi];
                    for (int a = 0; a < n_catoms; ++a)
                        tma_load_5d(sb + patch_bytes + (uint32_t)(j * n_catoms + a) * kDgWTile, &tmw, &full[st],
                                    c0 + 64 * a, tap, kc * 64, g, 0);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (whole warp)
        const uint32_t sbase = smem_u32(smem);
        const uint32_t sbo = (uint32_t)((p.bw == 8 ? p.PW : 8) * 128);
        const uint32_t idesc = p.idesc;
        int st = 0;
        uint32_t par = 0;
        for (int i = 0; i < nk; ++i) {
            if (!mbar_wait(&full[st], par)) break;
            tc_fence_after();
            const int tg = i % n_tg;
            const int y0 = tg * TG, ntap = min(TG, nyx - y0);
            const uint32_t sst = sbase + (uint32_t)(st * stage_bytes);
            for (int j = 0; j < ntap; ++j) {
                const int yi = (y0 + j) / nx, xi = (y0 + j) - yi * nx;
                const int shift = DH.shift[ph][yi] * p.PW + DW.shift[pw][xi];
                const uint64_t a0 = make_sdesc(sst + (uint32_t)shift * 128u, 16u, sbo, 2u, 0u);
                const uint64_t b0 =
                    make_sdesc(sst + (uint32_t)patch_bytes + (uint32_t)(j * n_catoms) * kDgWTile, kDgWTile, 1024u, 2u, 0u);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t acc = (i | j | ks) != 0 ? 1u : 0u;
                    if (elect_one()) umma_f16(tbase, a0 + (uint64_t)(2 * ks), b0 + (uint64_t)(128 * ks), idesc, acc);
                    __syncwarp();
                }
            }
            if (elect_one()) umma_commit(&empty[st]);
            __syncwarp();
            if (++st == stages) st = 0, par ^= 1u;
        }
        if (nk > 0 && elect_one()) umma_commit(accb);
        __syncwarp();
    }
    // ---------------------------------------------------- epilogue (all warps)
    named_bar_sync(2, kDgThreads);
    tc_fence_after();
    tbase = *tslot;
    {
        if (nk > 0) {
            mbar_wait_sleep(accb, 0);
            tc_fence_after();
        }
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const int jw = j0w + row % p.bw, jh = j0h + row / p.bw;
        const bool valid = jw < DW.J[pw] && jh < DH.J[ph] && td < DD.J[pd];
        const int w = pw + DW.nph * jw, h = ph + DH.nph * jh, di = pd + DD.nph * td;
        const long long pix = (((long long)n * p.Di + di) * p.Hi + h) * p.Wi + w;
        const long long obase = pix * p.ch_pix + (long long)g * p.C + c0;
        const int cblk = g * p.C + c0;  // this tile's first channel in the pixel
        const int Nt = p.Nt;
        const int c_mid = ((Nt >> 1) + 31) & ~31;
        const int c_lo = warp < 4 ? 0 : c_mid, c_hi = warp < 4 ? min(c_mid, Nt) : Nt;
        const uint32_t trow = tbase + ((uint32_t)(q * 32) << 16);
        for (int cb = c_lo; cb < c_hi; cb += 32) {
            float v[32];
            if (nk > 0) {
                dg_ld(trow + (uint32_t)cb, min(32, c_hi - cb), v);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
            }
            if (!valid) continue;
#pragma unroll
            for (int j = 0; j < 32; j += 8)
                if (cb + j < c_hi && c0 + cb + j < p.C && cblk + cb + j < p.ch_lim)
                    store8(p.out, obase + cb + j, v + j, p.out_dtype);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, (uint32_t)p.tmem_cols);
    }
}

}  // namespace wg
