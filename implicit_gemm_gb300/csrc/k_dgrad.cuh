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
//  * fp32 accumulators in TMEM, two buffers; warps 2..5 read them (one TMEM
//    lane quadrant, i.e. 32 pixels, per warp) and store dX.
//
// Warp roles (192 threads): warp 0 lane 0 issues TMA into an mbarrier ring,
// warp 1 issues the MMAs, warps 2..5 run the epilogue while the next tile's
// loads and MMAs proceed; every wait is bounded.
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
    int n_tw, n_th, n_td, N, n_ctiles;
    int n_all;          // tiles over phases, boxes, depth, images, channel tiles and group blocks (< 2^31)
    int T;              // taps of the filter (Z*Y*X)
    int w_resident;     // 1: every W tile stays in shared memory; the ring holds dY patches only
    int w_bytes;        // bytes of the resident W tiles
    int patch_bytes, stage_bytes, stages, tmem_cols;
    uint32_t idesc;
    int out_dtype;  // wg_dtype of dX
    void* out;
    DgDim dim[3];   // stride phases along (w, h, d): positions, dY offsets, taps and their row shifts
};

constexpr int kDgThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue (one TMEM lane quadrant each)
constexpr int kDgEpiWarps = 4;
constexpr int kDgMaxStages = 4;
// Epilogue staging: per epilogue warp 32 pixels x 64 bytes (one round of 32
// 16-bit or 16 fp32 channels), so that the global stores go out as 64-byte runs
// of one pixel instead of 16-byte pieces of 32 pixels.
constexpr int kDgStageRow = 64;
constexpr int kDgStagingBytes = kDgEpiWarps * 32 * kDgStageRow;
constexpr uint32_t kDgWTile = 8192;  // one W tile: 64 k rows x 64 c

// Pack 16 bytes of output: 4 fp32 values, or 8 values rounded to bf16/fp16.
__device__ __forceinline__ uint4 pack16(const float* v, int out_dtype)
{
    uint4 u;
    if (out_dtype == 2) {
        u.x = __float_as_uint(v[0]), u.y = __float_as_uint(v[1]);
        u.z = __float_as_uint(v[2]), u.w = __float_as_uint(v[3]);
        return u;
    }
    uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (out_dtype == 0) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
            w[j] = *reinterpret_cast<const uint32_t*>(&h);
        } else {
            const __half2 h = __floats2half2_rn(v[2 * j], v[2 * j + 1]);
            w[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
    }
    return u;
}

// Byte offset of 16-byte chunk k of pixel row r in a warp's staging buffer
// (32 rows of 64 bytes): the chunk index is XORed with (r / 2) % 4 so that
// both the row-wise writes and the chunk-wise reads are free of bank conflicts.
__device__ __forceinline__ uint32_t stg_off(int r, int k)
{
    return (uint32_t)(r * kDgStageRow + ((k ^ ((r >> 1) & 3)) << 4));
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
    // A programmatic dependent of the kernel before it (which may still read
    // the previous contents of `we`); the backward-data kernel launched after
    // it waits for this grid before it reads `we`.
    pdl_wait();
    pdl_launch_dependents();
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

// One tile of the persistent walk: stride phase (pw, ph, pd), box (tw, th) of
// phase positions, depth position td, image n, channel tile ct and group block g,
// with the phase's tap counts and the tile's stage count nk (0: no position of
// the box is in its phase, or no tap reaches the phase -- the tile is zeros).
struct DgTile {
    int pw, ph, pd, tw, th, td, n, ct, g;
    int nx, nz, nyx, n_tg, nk;
};

__device__ __forceinline__ DgTile dg_tile(const DgParams& p, int t)
{
    DgTile r;
    const DgDim& DW = p.dim[0];
    const DgDim& DH = p.dim[1];
    const DgDim& DD = p.dim[2];
    r.pw = (int)(t % DW.nph);
    t /= DW.nph;
    r.ph = (int)(t % DH.nph);
    t /= DH.nph;
    r.pd = (int)(t % DD.nph);
    t /= DD.nph;
    r.tw = (int)(t % p.n_tw);
    t /= p.n_tw;
    r.th = (int)(t % p.n_th);
    t /= p.n_th;
    r.td = (int)(t % p.n_td);
    t /= p.n_td;
    r.n = (int)(t % p.N);
    t /= p.N;
    r.ct = (int)(t % p.n_ctiles);
    r.g = (int)(t / p.n_ctiles);
    r.nx = DW.ntap[r.pw];
    r.nz = DD.ntap[r.pd];
    r.nyx = r.nx * DH.ntap[r.ph];
    r.n_tg = (r.nyx + p.TG - 1) / p.TG;
    const bool any = r.tw * p.bw < DW.J[r.pw] && r.th * p.bh < DH.J[r.ph] && r.td < DD.J[r.pd];
    r.nk = any ? p.n_kc * r.nz * r.n_tg : 0;
    return r;
}

// Persistent: CTA b takes tiles b, b + grid, b + 2 grid, ...  The stage ring
// runs on across tiles (the next tile's loads overlap this tile's MMAs) and the
// accumulator alternates between two TMEM buffers (the epilogue of one tile
// overlaps the MMAs of the next).
__global__ void __launch_bounds__(kDgThreads, 1)
    dgrad_kernel(const __grid_constant__ CUtensorMap tmy, const __grid_constant__ CUtensorMap tmw,
                 const __grid_constant__ DgParams p)
{
    extern __shared__ uint8_t smem_raw[];
    // [resident W tiles][ring of stages][epilogue staging][barriers]
    uint8_t* wres = align_shared<uint8_t>(smem_raw, 1024);
    uint8_t* smem = wres + p.w_bytes;
    uint8_t* staging = smem + p.stages * p.stage_bytes;
    uint8_t* tail = staging + kDgStagingBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(tail);
    uint64_t* empty = full + kDgMaxStages;
    uint64_t* accf = empty + kDgMaxStages;  // [2] accumulator b complete (MMA -> epilogue)
    uint64_t* acce = accf + 2;              // [2] accumulator b drained (epilogue -> MMA)
    uint64_t* wbar = acce + 2;              // the resident W tiles have landed
    uint32_t* tslot = reinterpret_cast<uint32_t*>(wbar + 1);
    const bool wr = p.w_resident != 0;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const DgDim& DW = p.dim[0];
    const DgDim& DH = p.dim[1];
    const DgDim& DD = p.dim[2];
    const int n_all = p.n_all;
    const int stages = p.stages, stage_bytes = p.stage_bytes, patch_bytes = p.patch_bytes;
    const int n_catoms = p.n_catoms, X = p.X, TG = p.TG, Nt = p.Nt;

    // The next kernel on the stream may be scheduled at once (it waits for this
    // grid before it reads what this grid writes).
    pdl_launch_dependents();
    // Thread 0 (the TMA producer) prefetches the tensor maps, initialises the
    // barriers and issues the resident W tiles before the block barrier, and
    // warp 1 allocates TMEM meanwhile: the TMA unit's first fetch of the
    // tensor maps then overlaps the prologue.  This kernel is a programmatic
    // dependent of the kernel before it: dY and W are read, and TMEM taken,
    // only after griddepcontrol.wait.
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmy);
        tma_prefetch_desc(&tmw);
        for (int i = 0; i < stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], kDgEpiWarps);
        }
        mbar_init(wbar, 1);
        fence_mbar_init();
        pdl_wait();
        if (wr) {
            // Every (K chunk, tap, channel atom) tile of the one (channel tile, group).
            mbar_arrive_expect_tx(wbar, (uint32_t)p.w_bytes);
            for (int kc = 0; kc < p.n_kc; ++kc)
                for (int tap = 0; tap < p.T; ++tap)
                    for (int a = 0; a < n_catoms; ++a)
                        tma_load_5d(wres + (uint32_t)((kc * p.T + tap) * n_catoms + a) * kDgWTile, &tmw, wbar,
                                    64 * a, tap, kc * 64, 0, 0);
        }
    }
    if (warp == 1) {
        pdl_wait();
        tmem_alloc(tslot, (uint32_t)p.tmem_cols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();  // barriers initialised, TMEM allocated, W on its way
    uint32_t tbase = 0;
    if (warp != 0) {
        tc_fence_after();
        tbase = *tslot;
    }

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            const uint32_t patch_tx = (uint32_t)(p.PW * p.PH * 128);
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_all && ok; t += gridDim.x) {
                const DgTile d = dg_tile(p, t);
                const int c0 = d.ct * Nt;
                for (int i = 0; i < d.nk; ++i, ++it) {
                    const int st = it % stages;
                    const uint32_t par = (uint32_t)(it / stages) & 1u;
                    if (it >= stages && !mbar_wait(&empty[st], par ^ 1u)) {
                        ok = false;
                        break;
                    }
                    const int tg = i % d.n_tg, rest = i / d.n_tg;
                    const int zi = rest % d.nz, kc = rest / d.nz;
                    const int y0 = tg * TG, ntap = min(TG, d.nyx - y0);
                    const int z = DD.tap[d.pd][zi];
                    uint8_t* sb = smem + st * stage_bytes;
                    mbar_arrive_expect_tx(&full[st], patch_tx + (wr ? 0u : (uint32_t)(ntap * n_catoms) * kDgWTile));
                    // The dY rows the box's positions read for every (y, x) tap of plane z.
                    tma_load_5d(sb, &tmy, &full[st], d.g * p.K + kc * 64, d.tw * p.bw + DW.qmin[d.pw],
                                d.th * p.bh + DH.qmin[d.ph], d.td + DD.qmin[d.pd] + DD.shift[d.pd][zi], d.n);
                    for (int j = 0; j < ntap && !wr; ++j) {
                        const int yi = (y0 + j) / d.nx, xi = (y0 + j) - yi * d.nx;
                        const int tap = (z * p.Y + DH.tap[d.ph][yi]) * X + DW.tap[d.pw][xi];
                        for (int a = 0; a < n_catoms; ++a)
                            tma_load_5d(sb + patch_bytes + (uint32_t)(j * n_catoms + a) * kDgWTile, &tmw, &full[st],
                                        c0 + 64 * a, tap, kc * 64, d.g, 0);
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (whole warp)
        const uint32_t sbase = smem_u32(smem), wbase = smem_u32(wres);
        const uint32_t sbo = (uint32_t)((p.bw == 8 ? p.PW : 8) * 128);
        const uint32_t idesc = p.idesc;
        int it = 0, u = 0;
        bool ok = !wr || mbar_wait(wbar, 0);
        for (int t = blockIdx.x; t < n_all && ok; t += gridDim.x) {
            const DgTile d = dg_tile(p, t);
            if (d.nk == 0) continue;
            const int b = u & 1;
            if (u >= 2 && !mbar_wait(&acce[b], (uint32_t)((u >> 1) - 1) & 1u)) break;
            tc_fence_after();
            const uint32_t tacc = tbase + (uint32_t)(b * Nt);
            for (int i = 0; i < d.nk; ++i, ++it) {
                const int st = it % stages;
                const uint32_t par = (uint32_t)(it / stages) & 1u;
                if (!mbar_wait(&full[st], par)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int tg = i % d.n_tg, rest = i / d.n_tg;
                const int zi = rest % d.nz, kc = rest / d.nz;
                const int y0 = tg * TG, ntap = min(TG, d.nyx - y0);
                const int z = DD.tap[d.pd][zi];
                const uint32_t sst = sbase + (uint32_t)(st * stage_bytes);
                // Descriptors are a base plus byte offsets added to the start-address
                // field (shared-memory addresses stay below 2^18, so the 14-bit field
                // never carries into the next one), and the tap's (y, x) index runs
                // as a counter: rebuilding both from the tap geometry for every tap
                // held back the MMA issue rate.
                const uint64_t a_base = make_sdesc(sst, 16u, sbo, 2u, 0u);
                const uint64_t b_base = wr ? make_sdesc(wbase, kDgWTile, 1024u, 2u, 0u)
                                           : make_sdesc(sst + (uint32_t)patch_bytes, kDgWTile, 1024u, 2u, 0u);
                const int ztap = z * p.Y;
                const int kcT = kc * p.T;
                int yi = y0 / d.nx, xi = y0 - yi * d.nx;
                for (int j = 0; j < ntap; ++j) {
                    const int shift = DH.shift[d.ph][yi] * p.PW + DW.shift[d.pw][xi];
                    const uint64_t a0 = a_base + (uint64_t)(shift * 8);  // 128 bytes per row, in 16-byte units
                    // B: this tap's W tile -- resident (indexed by K chunk and tap) or in the stage.
                    const int tap = (ztap + DH.tap[d.ph][yi]) * X + DW.tap[d.pw][xi];
                    const int wt = wr ? (kcT + tap) * n_catoms : j * n_catoms;
                    const uint64_t b0 = b_base + (uint64_t)(wt * (kDgWTile >> 4));
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint32_t acc = (i | j | ks) != 0 ? 1u : 0u;
                        if (elect_one()) umma_f16(tacc, a0 + (uint64_t)(2 * ks), b0 + (uint64_t)(128 * ks), idesc, acc);
                        __syncwarp();
                    }
                    if (++xi == d.nx) xi = 0, ++yi;
                }
                if (elect_one()) umma_commit(&empty[st]);
                __syncwarp();
            }
            if (!ok) break;
            if (elect_one()) umma_commit(&accf[b]);
            __syncwarp();
            ++u;
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        // Warp q drains TMEM lanes 32q..32q+31 (pixels of the box) in rounds of
        // 64 bytes per pixel: each lane converts its pixel's columns and writes
        // them to the warp's staging rows; then lane i stores chunk i % 4 of
        // pixels i / 4, 8 + i / 4, 16 + i / 4 and 24 + i / 4, so that a store
        // instruction covers eight 64-byte runs.  Tiles of zeros skip TMEM and
        // staging and store zeros in the same pattern.
        pdl_wait();  // returns at once: the previous kernel finished before the first load
        const int q = warp & 3;
        const uint32_t trow = tbase + ((uint32_t)(q * 32) << 16);
        const uint32_t sw = smem_u32(staging) + (uint32_t)(q * 32 * kDgStageRow);
        const int od = p.out_dtype;
        const int esz = od == 2 ? 4 : 2;
        const int cpr = kDgStageRow / esz;  // channels per round
        const int kq = lane & 3;            // this lane's chunk of a pixel's run
        const int kch = kq * (16 / esz);    // its first channel within the round
        int u = 0;
        for (int t = blockIdx.x; t < n_all; t += gridDim.x) {
            const DgTile d = dg_tile(p, t);
            const int c0 = d.ct * Nt;
            const int cblk = d.g * p.C + c0;  // this tile's first channel in the pixel
            long long obase[4];
            bool valid[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int row = q * 32 + r * 8 + (lane >> 2);
                const int jw = d.tw * p.bw + row % p.bw, jh = d.th * p.bh + row / p.bw;
                valid[r] = jw < DW.J[d.pw] && jh < DH.J[d.ph] && d.td < DD.J[d.pd];
                const int w = d.pw + DW.nph * jw, h = d.ph + DH.nph * jh, di = d.pd + DD.nph * d.td;
                const long long pix = (((long long)d.n * p.Di + di) * p.Hi + h) * p.Wi + w;
                obase[r] = pix * p.ch_pix + cblk;
            }
            const int b = u & 1;
            const bool have = d.nk > 0;
            if (have) {
                if (!mbar_wait_sleep(&accf[b], (uint32_t)(u >> 1) & 1u)) break;
                tc_fence_after();
            }
            for (int cb = 0; cb < Nt; cb += cpr) {
                uint4 val = make_uint4(0u, 0u, 0u, 0u);
                if (have) {
                    float v[32];
                    dg_ld(trow + (uint32_t)(b * Nt + cb), min(cpr, Nt - cb), v);
                    uint4 c[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) c[k] = od == 2 ? pack16(v + 4 * k, 2) : pack16(v + 8 * k, od);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sw + stg_off(lane, k)),
                                     "r"(c[k].x), "r"(c[k].y), "r"(c[k].z), "r"(c[k].w)
                                     : "memory");
                    __syncwarp();
                }
                // Channels are checked in groups of 8 (the layout's granularity).
                const int g8 = (cb + kch) & ~7;
                const bool ch_ok = cb + kch < Nt && c0 + g8 < p.C && cblk + g8 < p.ch_lim;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int px = r * 8 + (lane >> 2);
                    if (have)
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                                     : "r"(sw + stg_off(px, kq))
                                     : "memory");
                    if (valid[r] && ch_ok) {
                        uint8_t* o = static_cast<uint8_t*>(p.out) + (obase[r] + cb + kch) * esz;
                        *reinterpret_cast<uint4*>(o) = val;
                    }
                }
                if (have) __syncwarp();  // the next round overwrites the staging rows
            }
            if (have) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acce[b]);
                ++u;
            }
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
