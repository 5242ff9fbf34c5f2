// Tensor-core implicit-GEMM weight gradient (sm_103a: TMA + tcgen05 + TMEM).
//
// The GEMM of "Composable Kernel: grouped_convolution_backward_weight_kernel.hpp
// Source File" (GroupedConvBwdWeightKernelArgs: GemmM = K, GemmN = C*YX,
// GemmK = N*Ho*Wo, batched over G via the group strides; grid = (tiles, G,
// k_batch) in GridSize / operator()) is computed here as its transpose
//
//     D[(tap, c), k] = sum over pixels p of Xcol[p, (tap, c)] * dY[p, k]
//
// so that the long (tap, c) axis sits on the 128 MMA rows and the output
// channels k on the MMA N columns.  Both operands are staged in shared memory
// with the free axis contiguous and the reduction axis (pixels) strided -- the
// "K-outer" arrangement that PR #11602 ("add transpose load for bwd weight and
// bwd data") describes for gfx950 -- which tcgen05 consumes directly as
// MN-major operands (128-byte swizzle), so nothing is ever transposed.
//
// X staging (chosen by the planner):
//  * halo: one TMA box per (stride phase, 64-channel chunk) covers every tap
//    of a K-tile of output pixels; the A operand of tap (z,y,x) is the same
//    patch read from a row offset (shared-memory descriptors are
//    address-swizzled, so any 128-byte row offset is a valid start).
//  * per-tap: one TMA box per (tap, chunk) with the tap offset in its
//    coordinates and the conv stride as the TMA element stride.
// Implicit zero padding is the TMA out-of-bounds fill, for both operands.
//
// Warp roles (192 threads): warp 0 lane 0 issues TMA; warp 1 owns TMEM and its
// lane 0 issues tcgen05.mma; warps 2..5 read TMEM (lane quadrant = warp % 4)
// and store dW / atomically add / write the split-K workspace.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "ptx.cuh"

namespace wg {

// Most M-tiles one CTA accumulates (TMEM columns = M-tiles x Nt <= 512).
constexpr int kMaxMt = 16;

struct IgParams {
    int G, C, K, T, GC, GK;
    int X, Y;                // filter extents along w and h (tap = (z*Y + y)*X + x)
    int ncc;                 // 64-channel chunks per tap
    int s[3], d[3], pl[3];   // stride, dilation, left pad along (w, h, d)
    int box[4], ntile[4];    // pixel tile and tile counts along (w, h, d, n)
    int KT, ksteps;
    int per_split, total_kt;
    int Gm, Nt, n_ntiles, n_katoms, n_atoms, n_mtiles, mtpc;
    int halo;
    int patch[3];
    int patch_bytes, patch_tx;
    int n_patches, dy_off, slot_bytes, stage_bytes, stages;
    int tmem_cols;
    uint32_t idesc;
    int mode;       // 1 direct, 2 atomic, 3 workspace
    int out_dtype;  // wg_dtype
    void* out;
    long long split_stride;
    unsigned char patch_ph[32][4];
    unsigned int atom_off[256];
    unsigned short atom_tap[256];
    unsigned char atom_cc[256];
};

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Epilogue of one M-tile for one warp: TMEM -> registers -> global, in chunks
// of 16 columns.  MODE 1 stores dW in OUT (fp32, bf16 or fp16), MODE 2 adds
// to fp32 dW with global atomics, MODE 3 stores fp32 to the split's workspace
// slice.  Each lane owns one row (tap, c); k runs over the chunk's columns.
template <int MODE, typename OUT>
__device__ __forceinline__ void epilogue_mtile(uint32_t taddr, int ncols, bool have_acc, bool vrow, int n_lo, int K,
                                               OUT* __restrict__ out, long long rowbase, long long kstride)
{
    for (int c16 = 0; c16 < ncols; c16 += 16) {
        float v[16];
        if (have_acc) {
            tmem_ld16(taddr + (uint32_t)c16, v);
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = 0.f;
        }
        if (!vrow) continue;
        const int k0 = c16 - n_lo;
        OUT* o = out + rowbase + (long long)k0 * kstride;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int k = k0 + j;
            if (k >= 0 && k < K) {
                if constexpr (MODE == 2) {
                    red_add_f32(reinterpret_cast<float*>(o), v[j]);
                } else if constexpr (sizeof(OUT) == 4) {
                    *o = v[j];
                } else if constexpr (sizeof(OUT) == 2 && std::is_same<OUT, __nv_bfloat16>::value) {
                    *o = __float2bfloat16_rn(v[j]);
                } else {
                    *o = __float2half_rn(v[j]);
                }
            }
            o += kstride;
        }
    }
}

// The MMA issuer, run by a whole converged warp so that every operand is
// warp-uniform: descriptors are sums of 64-bit parts whose fields never
// overlap -- the M-tile part (start of its first atom in stage 0, LBO to its
// second atom), the K-step part (row offset of the step's first 8-pixel group
// in the start field, SBO to its second group) and the stage offset -- formed
// from kernel parameters and loop counters only, and one elected lane issues a
// K-step's MT MMAs (MT a compile-time count, fully unrolled).
struct MmaArgs {
    uint64_t b0;        // dY descriptor of stage 0, K-step 0
    uint32_t idesc, Nt, stage16;
    int ksteps, stages, bw, bh, bd, PW, PH, PD;
    int linear;         // per-tap boxes: K-row r of a tile is box row r
};

template <int MT>
__device__ __forceinline__ void mma_mainloop(const MmaArgs a, const uint64_t (&ab)[kMaxMt], uint64_t* full,
                                             uint64_t* empty, uint64_t* accb, uint32_t tbase, int nk)
{
    const uint64_t b0 = a.b0;
    const uint32_t idesc = a.idesc, Nt = a.Nt, stage16 = a.stage16;
    const int ksteps = a.ksteps, stages = a.stages, bw = a.bw, bh = a.bh, bd = a.bd;
    const int PW = a.PW, PH = a.PH, PD = a.PD;
    const bool linear = a.linear != 0;
    int st = 0;
    uint32_t ph = 0;
    for (int i = 0; i < nk; ++i) {
        if (!mbar_wait(&full[st], ph)) break;
        tc_fence_after();
        const uint64_t soff = (uint64_t)((uint32_t)st * stage16);
        // Pixel coordinates (iw, ih, id, in) of the current 8-pixel group inside
        // the tile (w fastest), advanced group by group.
        int iw = 0, ih = 0, id = 0, in = 0;
        for (int ks = 0; ks < ksteps; ++ks) {
            uint32_t r0, r1;
            if (linear) {
                r0 = (uint32_t)(16 * ks);
                r1 = r0 + 8u;
            } else {
                // Halo patch: the tile's w extent is a multiple of 8, so each
                // 8-pixel group is one run of a patch row.
                r0 = (uint32_t)(((in * PD + id) * PH + ih) * PW + iw);
                iw += 8;
                if (iw >= bw) { iw = 0; if (++ih == bh) { ih = 0; if (++id == bd) { id = 0; ++in; } } }
                r1 = (uint32_t)(((in * PD + id) * PH + ih) * PW + iw);
                iw += 8;
                if (iw >= bw) { iw = 0; if (++ih == bh) { ih = 0; if (++id == bd) { id = 0; ++in; } } }
            }
            const uint64_t kd = ((uint64_t)((r1 - r0) * 8u) << 32) + (uint64_t)(r0 * 8u) + soff;
            const uint64_t bdesc = b0 + soff + (uint64_t)(ks * 128);
            const uint32_t acc = (i | ks) != 0 ? 1u : 0u;
            if (elect_one()) {
#pragma unroll
                for (int m = 0; m < MT; ++m) umma_f16(tbase + (uint32_t)m * Nt, ab[m] + kd, bdesc, idesc, acc);
            }
            __syncwarp();
        }
        if (elect_one()) umma_commit(&empty[st]);
        __syncwarp();
        if (++st == stages) st = 0, ph ^= 1u;
    }
    if (elect_one()) umma_commit(accb);
    __syncwarp();
}

__global__ void __launch_bounds__(192, 1)
    igemm_wgrad_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmy,
                       const __grid_constant__ IgParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // [stages x stage_bytes][1 KB slack read by padding atoms][tail: barriers + tables]
    uint8_t* tail = smem + p.stages * p.stage_bytes + 1024;
    uint64_t* full = reinterpret_cast<uint64_t*>(tail);
    uint64_t* empty = full + 8;
    uint64_t* accb = empty + 8;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(accb + 1);

    // Scalars used in loops are read into registers once here.
    const int Nt = p.Nt, ksteps = p.ksteps, stages = p.stages, stage_bytes = p.stage_bytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mr = blockIdx.x / p.n_ntiles, nt = blockIdx.x % p.n_ntiles;
    const int gb = blockIdx.y, split = blockIdx.z;
    const int kt0 = split * p.per_split;
    const int nk = max(0, min(p.per_split, p.total_kt - kt0));
    const int mt0 = mr * p.mtpc;
    const int mtn = min(p.mtpc, p.n_mtiles - mt0);
    const int atom0 = 2 * mt0;
    const int g0 = gb * p.Gm;
    const int c_al = (g0 * p.C) & ~7;
    const int k_base = ((g0 * p.K) & ~7) + nt * p.Nt;

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(accb, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, (uint32_t)p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
#define MMA_ARGS ma, ab, full, empty, accb, tbase, nk

    if (warp == 0) {
        if (lane == 0 && nk > 0) {
            // ------------------------------------------------ TMA producer
            tma_prefetch_desc(&tmx);
            tma_prefetch_desc(&tmy);
            const uint32_t tx = (uint32_t)(p.n_patches * p.patch_tx + p.n_katoms * p.slot_bytes);
            for (int i = 0; i < nk; ++i) {
                const int st = i % p.stages;
                const uint32_t ph = (uint32_t)(i / p.stages) & 1u;
                if (i >= p.stages && !mbar_wait(&empty[st], ph ^ 1u)) break;
                uint8_t* sb = smem + st * p.stage_bytes;
                mbar_arrive_expect_tx(&full[st], tx);
                int kt = kt0 + i;
                const int tw = kt % p.ntile[0];
                kt /= p.ntile[0];
                const int th = kt % p.ntile[1];
                kt /= p.ntile[1];
                const int td = kt % p.ntile[2];
                const int tn = kt / p.ntile[2];
                const int wo0 = tw * p.box[0], ho0 = th * p.box[1], do0 = td * p.box[2], n0 = tn * p.box[3];
                const int bw = wo0 * p.s[0] - p.pl[0], bh = ho0 * p.s[1] - p.pl[1], bd = do0 * p.s[2] - p.pl[2];
                if (p.halo) {
                    for (int q = 0; q < p.n_patches; ++q)
                        tma_load_5d(sb + q * p.patch_bytes, &tmx, &full[st], c_al + 64 * p.patch_ph[q][3],
                                    bw + p.patch_ph[q][0], bh + p.patch_ph[q][1], bd + p.patch_ph[q][2], n0);
                } else {
                    for (int a = 0; a < p.n_patches; ++a) {
                        const int atom = atom0 + a;
                        if (a < 2 * mtn && atom < p.n_atoms) {
                            const int tap = atom / p.ncc, cc = atom - tap * p.ncc;
                            const int x = tap % p.X, y = (tap / p.X) % p.Y, z = tap / (p.X * p.Y);
                            tma_load_5d(sb + a * p.patch_bytes, &tmx, &full[st], c_al + 64 * cc, bw + x * p.d[0],
                                        bh + y * p.d[1], bd + z * p.d[2], n0);
                        } else {
                            // Padding atom: a box entirely past the channel extent reads zeros.
                            tma_load_5d(sb + a * p.patch_bytes, &tmx, &full[st], p.GC, 0, 0, 0, 0);
                        }
                    }
                }
                for (int j = 0; j < p.n_katoms; ++j)
                    tma_load_5d(sb + p.dy_off + j * p.slot_bytes, &tmy, &full[st], k_base + 64 * j, wo0, ho0, do0, n0);
            }
        }
    } else if (warp == 1) {
        if (nk > 0) {
            // ------------------------------------------------ MMA issuer (whole warp)
            const uint32_t sbase = smem_u32(smem);
            uint64_t ab[kMaxMt];
#pragma unroll
            for (int m = 0; m < kMaxMt; ++m) {
                ab[m] = 0;
                if (m < mtn) {
                    const int a = atom0 + 2 * m;
                    uint32_t off_a, off_b;
                    if (p.halo) {
                        off_a = p.atom_off[a];
                        off_b = (a + 1 < p.n_atoms) ? p.atom_off[a + 1] : off_a + 1024u;
                    } else {
                        off_a = (uint32_t)(2 * m * p.patch_bytes);
                        off_b = off_a + (uint32_t)p.patch_bytes;
                    }
                    ab[m] = make_sdesc(sbase + off_a, off_b - off_a, 0u, 2u, 0u);
                }
            }
            MmaArgs ma;
            ma.b0 = make_sdesc(sbase + (uint32_t)p.dy_off, (uint32_t)p.slot_bytes, 1024u, 2u, 0u);
            ma.idesc = p.idesc, ma.Nt = (uint32_t)Nt, ma.stage16 = (uint32_t)stage_bytes >> 4;
            ma.ksteps = ksteps, ma.stages = stages, ma.bw = p.box[0], ma.bh = p.box[1], ma.bd = p.box[2];
            ma.PW = p.patch[0], ma.PH = p.patch[1], ma.PD = p.patch[2];
            ma.linear = p.halo ? 0 : 1;
            switch (mtn) {
                case 1: mma_mainloop<1>(MMA_ARGS); break;
                case 2: mma_mainloop<2>(MMA_ARGS); break;
                case 3: mma_mainloop<3>(MMA_ARGS); break;
                case 4: mma_mainloop<4>(MMA_ARGS); break;
                case 5: mma_mainloop<5>(MMA_ARGS); break;
                case 6: mma_mainloop<6>(MMA_ARGS); break;
                case 7: mma_mainloop<7>(MMA_ARGS); break;
                case 8: mma_mainloop<8>(MMA_ARGS); break;
                case 9: mma_mainloop<9>(MMA_ARGS); break;
                case 10: mma_mainloop<10>(MMA_ARGS); break;
                case 11: mma_mainloop<11>(MMA_ARGS); break;
                case 12: mma_mainloop<12>(MMA_ARGS); break;
                case 13: mma_mainloop<13>(MMA_ARGS); break;
                case 14: mma_mainloop<14>(MMA_ARGS); break;
                case 15: mma_mainloop<15>(MMA_ARGS); break;
                default: mma_mainloop<16>(MMA_ARGS); break;
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        if (nk > 0) {
            mbar_wait_sleep(accb, 0);
            tc_fence_after();
        }
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const int K = p.K, C = p.C, T = p.T, GC = p.GC, Gm = p.Gm, n_atoms = p.n_atoms, ncc = p.ncc, mode = p.mode;
        const int out_dtype = p.out_dtype;
        void* const out = p.out;
        const long long split_off = (long long)split * p.split_stride;
        const uint32_t trow = tbase + ((uint32_t)(q * 32) << 16);
        const bool have_acc = nk > 0;
        for (int m = 0; m < mtn; ++m) {
            const int atom = atom0 + 2 * m + (row >> 6);
            bool vrow = atom < n_atoms;
            int tap = 0, cc = 0;
            if (vrow) {
                if (p.halo) {
                    tap = p.atom_tap[atom];
                    cc = p.atom_cc[atom];
                } else {
                    tap = atom / ncc;
                    cc = atom - tap * ncc;
                }
            }
            const int cg = c_al + cc * 64 + (row & 63);
            const int gr = cg / C;
            const int c = cg - gr * C;
            vrow = vrow && cg < GC && gr >= g0 && gr < g0 + Gm;
            const int n_lo = gr * K - k_base;
            const long long rowbase = ((long long)gr * K * T + tap) * C + c;
            const long long kstride = (long long)T * C;
            const uint32_t ta = trow + (uint32_t)(m * Nt);
            if (mode == 3) {
                epilogue_mtile<3, float>(ta, Nt, have_acc, vrow, n_lo, K, static_cast<float*>(out) + split_off, rowbase,
                                         kstride);
            } else if (mode == 2) {
                if (have_acc)
                    epilogue_mtile<2, float>(ta, Nt, true, vrow, n_lo, K, static_cast<float*>(out), rowbase, kstride);
            } else if (out_dtype == 2) {
                epilogue_mtile<1, float>(ta, Nt, have_acc, vrow, n_lo, K, static_cast<float*>(out), rowbase, kstride);
            } else if (out_dtype == 0) {
                epilogue_mtile<1, __nv_bfloat16>(ta, Nt, have_acc, vrow, n_lo, K, static_cast<__nv_bfloat16*>(out),
                                                 rowbase, kstride);
            } else {
                epilogue_mtile<1, __half>(ta, Nt, have_acc, vrow, n_lo, K, static_cast<__half*>(out), rowbase, kstride);
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

// Stage 2 of the deterministic split-K mode (the two-stage wgrad that PR
// #11602 and PR #12359 refer to): dW = cast(sum over splits of ws[s]).  The
// summation order is fixed, so the result is bitwise reproducible: the S
// splits are cut into kRedLanes contiguous ranges, each range is summed in
// index order, then the range sums are added in range order.
constexpr int kRedLanes = 8;
constexpr int kRedVecs = 32;  // float4 groups per CTA

__device__ __forceinline__ void store4(void* dw, long long i4, float4 a, int out_dtype)
{
    if (out_dtype == 2) {
        reinterpret_cast<float4*>(dw)[i4] = a;
    } else if (out_dtype == 0) {
        __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(dw) + 2 * i4;
        o[0] = __floats2bfloat162_rn(a.x, a.y);
        o[1] = __floats2bfloat162_rn(a.z, a.w);
    } else {
        __half2* o = reinterpret_cast<__half2*>(dw) + 2 * i4;
        o[0] = __floats2half2_rn(a.x, a.y);
        o[1] = __floats2half2_rn(a.z, a.w);
    }
}

// blockDim = (kRedVecs, kRedLanes).  E % 4 == 0: float4 groups; otherwise the
// same code on single floats (x, y, z, w of a float4 all used only in slot x).
__global__ void __launch_bounds__(kRedVecs* kRedLanes)
    reduce_splits_kernel(const float* __restrict__ ws, void* __restrict__ dw, long long E, int S, int out_dtype)
{
    __shared__ float4 part[kRedLanes][kRedVecs];
    const bool vec = (E & 3) == 0;
    const long long n = vec ? E / 4 : E;
    const long long i = (long long)blockIdx.x * kRedVecs + threadIdx.x;
    const int lane = threadIdx.y;
    const int L = (S + kRedLanes - 1) / kRedLanes;
    const int s0 = lane * L, s1 = min(S, s0 + L);
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < n) {
        if (vec) {
            const float4* w4 = reinterpret_cast<const float4*>(ws);
            int s = s0;
            for (; s + 4 <= s1; s += 4) {
                const float4 v0 = w4[(long long)s * n + i], v1 = w4[(long long)(s + 1) * n + i];
                const float4 v2 = w4[(long long)(s + 2) * n + i], v3 = w4[(long long)(s + 3) * n + i];
                a.x += v0.x, a.y += v0.y, a.z += v0.z, a.w += v0.w;
                a.x += v1.x, a.y += v1.y, a.z += v1.z, a.w += v1.w;
                a.x += v2.x, a.y += v2.y, a.z += v2.z, a.w += v2.w;
                a.x += v3.x, a.y += v3.y, a.z += v3.z, a.w += v3.w;
            }
            for (; s < s1; ++s) {
                const float4 v = w4[(long long)s * n + i];
                a.x += v.x, a.y += v.y, a.z += v.z, a.w += v.w;
            }
        } else {
            for (int s = s0; s < s1; ++s) a.x += ws[(long long)s * n + i];
        }
    }
    part[lane][threadIdx.x] = a;
    __syncthreads();
    if (lane == 0 && i < n) {
        float4 r = part[0][threadIdx.x];
        for (int l = 1; l < kRedLanes; ++l) {
            const float4 b = part[l][threadIdx.x];
            r.x += b.x, r.y += b.y, r.z += b.z, r.w += b.w;
        }
        if (vec) {
            store4(dw, i, r, out_dtype);
        } else if (out_dtype == 2) {
            static_cast<float*>(dw)[i] = r.x;
        } else if (out_dtype == 0) {
            static_cast<__nv_bfloat16*>(dw)[i] = __float2bfloat16_rn(r.x);
        } else {
            static_cast<__half*>(dw)[i] = __float2half_rn(r.x);
        }
    }
}

}  // namespace wg
