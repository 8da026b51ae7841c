// Exact INT8 GEMM of the W8A8 Linear on the sm_103a tensor cores.
//
// "TurboDiffusion Integration Notes", section "Differences From
// TurboDiffusion": the post-scale kernel keeps the integer accumulation
// continuous across K and applies the activation and weight scales in the
// epilogue; TurboDiffusion's original kernel is blockwise-scaled.  Both
// modes are computed here.
//
// GB300 has no 8-bit integer tcgen05 MMA (kind::i8 does not assemble for
// sm_103a), so the integer product runs on the bf16 pipe (kind::f16) with
// fp32 accumulation in tensor memory, which is exact for this data:
//   - every int8 value in [-127, 127] is exact in bf16, and every product
//     (|p| <= 16129) is exact in fp32;
//   - a chunk of at most 1024 K has a sum of absolute products of at most
//     127*127*1024 = 16,516,096 < 2^24, so every partial sum, in any order
//     and with any alignment of the addends, is an integer that fp32 holds
//     exactly;
//   - after each chunk the fp32 accumulator is read out of tensor memory
//     and added into an int32 running sum held in registers.
// The post-scale mode folds every 1024 K (16 stages of 64); the blockwise
// mode folds at every 128-wide K block, where the fp32 value read out is the
// block's exact integer partial P, and applies acc = acc + (P * sx) * sw.
//
// Kernel layout: clusters of two CTAs (one per SM), persistent over output
// tiles of 256 rows x BN columns (BN = 256, 224 or 192, chosen per shape).
// The pair shares each tile: CTA r loads rows [128r, 128r+128) of the A tile
// and rows [r*BN/2, (r+1)*BN/2) of the B tile into its own shared memory.
//   warp 0       TMA producer (both CTAs): bf16 A and B stages, 128-byte
//                swizzle, 6- or 7-deep ring; completion is counted on the leader's
//                barrier;
//   warp 1       TMEM allocator (both CTAs) and, in the leader only, the MMA
//                issuer: tcgen05.mma.cta_group::2 (M = 256, N = BN) into one
//                of two BN-column fp32 accumulators in each CTA's TMEM,
//                commits multicast to both CTAs;
//   warps 4..11  epilogue (both CTAs): each warp reads its 32 TMEM lanes
//                (rows) x BN/2 columns, folds chunks into registers, writes
//                the output with scales and bias, and releases the buffer
//                with a remote arrive on the leader's barrier.
// Two accumulator buffers let the MMA of chunk c+1 run while chunk c is
// folded.
//
// Variants of the same kernel (each described where it is defined):
//   - few tokens (M <= 256, post-scale): operands swapped so the weight rows
//     take the 256-row side and the tokens the N side (32..256), Y written
//     transposed; with few weight tiles, K split into units whose exact
//     int32 partials a finalize kernel sums (store_swapped, store_partial,
//     splitk_finalize_kernel);
//   - FFN up-projection: the epilogue applies GELU and the 1x128
//     quantization of the down-projection's input, staged through shared
//     memory over the next tile's chunk folds (stage_y, gelu_slice);
//   - few tokens on int8 operands (M <= 288): single-CTA kernels that
//     stream the int8 weight codes, widen them into tensor memory and
//     multiply them with an fp16 image of the tokens (gemm_s8.cu).
// Every kernel triggers its dependents' launch at its start and waits on
// its own prerequisite grid after its prologue (programmatic dependent
// launch); weights packed before the previous kernel started may be read
// before that wait.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdio>

#include "gelu.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "quant_core.cuh"

namespace w8a8 {
namespace {

constexpr int BM = 128;  // rows of A per CTA; a CTA pair covers TILE_M rows
constexpr int TILE_M = 2 * BM;
constexpr int BK = 64;   // bf16 elements per stage row = 128 bytes = one swizzle row
constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr uint32_t MAX_DYN_SMEM = 232448;  // 227 KB opt-in shared memory per block
// Output staging for the TMA-store epilogue: per epilogue warp, two 1 KB
// buffers of 32 rows x 16 bf16 columns (32-byte swizzle).
constexpr uint32_t STAGE_OUT_BYTES = 32 * 16 * 2;
constexpr int OUT_BUFS = 1;  // staging buffers per epilogue warp
constexpr uint32_t STAGING_BYTES = 8 * OUT_BUFS * STAGE_OUT_BYTES;
constexpr uint32_t RING_BUDGET = MAX_DYN_SMEM - 1024 - 256 - 512 - STAGING_BYTES;
constexpr int EPI_WARPS = 8;
constexpr int EPI_WARP0 = 4;  // warps 0-3: producer, MMA issuer, two idle; warps 4-11: epilogue
constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
// Register split (setmaxnreg): launched at 168 per thread (384 x 168 = 64512),
// warpgroup 0 drops to 56 and the two epilogue warpgroups rise to 224:
// 128 x 56 + 256 x 224 = 64512.
constexpr int REGS_LOW = 56;
constexpr int REGS_HIGH = 224;
static_assert(128 * REGS_LOW + 256 * REGS_HIGH <= THREADS * 168, "register split exceeds the launch budget");
constexpr uint32_t TMEM_COLS = 512;
constexpr int POSTSCALE_CHUNK_STAGES = 16;  // 1024 K: 127*127*1024 < 2^24
constexpr int BLOCK_CHUNK_STAGES = 2;       // one 128-wide scale block
// Tile raster: consecutive tiles walk the row tiles of a band of group_m row
// tiles (a KParams value) before moving to the next column tile, so a band's
// A rows stay in L2 while the B columns stream past.  The post-scale GEMM
// takes bands of 16 row tiles (4096 rows: the weight image is read once per
// band, and a band of A is 42 MB at K = 5120); the blockwise GEMM keeps 8.
constexpr int GROUP_M_POSTSCALE = 16;
constexpr int GROUP_M_BLOCKWISE = 8;
constexpr int SCALE_PREFETCH = 4;           // blockwise: per-block scales loaded this many chunks ahead
constexpr int kSwapMaxTokens = 256;         // post-scale GEMMs with M <= this swap operands
constexpr int kInt8MaxTokens = 288;         // post-scale GEMMs with M <= this can stream int8 operands
constexpr int kSplitTargetUnits = 72;       // split K until about this many CTA-pair work units exist
constexpr int kSplitMinStages = 4;          // at least 256 K per split
constexpr int kSplitMax = 8;

// Shared memory of the FFN up-projection's staged GELU input: one bf16 row
// of 128 columns per epilogue thread (8 warps x 32 rows x 256 bytes).
constexpr uint32_t YSTAGE_BYTES = EPI_WARPS * 32 * 256;

// Per-tile-width constants; EXTRA bytes of shared memory are taken from the ring.
template <int BN_, uint32_t EXTRA = 0>
struct Cfg {
    static constexpr int BN = BN_;
    static constexpr int HALF = BN / 2;  // B rows per CTA = output columns per epilogue warp
    static_assert(HALF % 16 == 0 && BN <= 256, "tile width");
    static constexpr uint32_t B_BYTES = HALF * BK * 2;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t RING = RING_BUDGET - EXTRA;
    static constexpr int STAGES = (RING / STAGE_BYTES) > 8 ? 8 : int(RING / STAGE_BYTES);
    static constexpr size_t SMEM = 1024 + size_t(STAGES) * STAGE_BYTES + STAGING_BYTES + EXTRA + 256;
    static constexpr uint32_t IDESC = idesc_bf16_f32(TILE_M, BN);
    static constexpr int LDW = (HALF % 32 == 0) ? 32 : 16;  // TMEM load width (columns)
    static constexpr int GROUPS = HALF / LDW;
};

enum WaitSite : int {
    kSiteProducerEmpty = 1,
    kSiteMmaAccEmpty = 2,
    kSiteMmaFull = 3,
    kSiteEpiAccFull = 4,
    kSiteMmaDrain = 5,
    kSiteProducerDrain = 6,
};

struct KParams {
    const float* sx;
    const float* sw;
    const __nv_bfloat16* bias;
    void* out;
    int M, N, K;
    int num_m, num_n, num_tiles;
    int k_stages, chunk_stages, kb_count;
    int tma_store;  // bf16 output written through shared memory and TMA (needs N % 8 == 0)
    int k_split;    // work units per tile, each over split_stages K stages (1: no split)
    int split_stages;
    int32_t* partial;  // k_split > 1: int32 partial sums [k_split][N][M] in kernel dims
    float* sg;         // kEpiGeluQuant: block scales [M][N/128]
    int a_settled;     // operand A (resp. B) was complete before the previous kernel in the
    int b_settled;     // stream started, so it may be read before the grid dependency wait
    int group_m;       // row tiles per raster band
};

__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int group_m, int& mb, int& nb) {
    const int per_group = group_m * num_n;
    const int group = tile / per_group;
    const int first_m = group * group_m;
    const int gm = min(num_m - first_m, group_m);
    const int local = tile - group * per_group;
    mb = first_m + local % gm;
    nb = local / gm;
}

// One work unit: a tile and the K stages [ks0, ks1) it accumulates.
struct Unit {
    int mb, nb, split, ks0, ks1;
};

__device__ __forceinline__ Unit unit_coords(int u, const KParams& p) {
    Unit w;
    const int tile = u / p.k_split;
    w.split = u - tile * p.k_split;
    tile_coords(tile, p.num_m, p.num_n, p.group_m, w.mb, w.nb);
    w.ks0 = w.split * p.split_stages;
    w.ks1 = min(p.k_stages, w.ks0 + p.split_stages);
    return w;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

template <int EPI>
struct AccType {
    using T = int32_t;
};
template <>
struct AccType<kEpiBlockwiseBf16> {
    using T = float;
};
template <>
struct AccType<kEpiBlockwiseF32> {
    using T = float;
};

template <int W>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[W]);
template <>
__device__ __forceinline__ void tmem_ld_cols<16>(uint32_t taddr, uint32_t (&r)[16]) {
    tmem_ld_32x32b_x16(taddr, r);
}
template <>
__device__ __forceinline__ void tmem_ld_cols<32>(uint32_t taddr, uint32_t (&r)[32]) {
    tmem_ld_32x32b_x32(taddr, r);
}
__device__ __forceinline__ void tmem_wait_cols(uint32_t (&r)[16]) { tmem_wait_ld_regs(r); }
__device__ __forceinline__ void tmem_wait_cols(uint32_t (&r)[32]) { tmem_wait_ld_regs32(r); }

// Write the COLS accumulated columns [col0, col0+COLS) of one row.  The
// per-column scales and bias are read through the read-only path (they never
// alias Y), so their loads need not wait behind this row's stores.
template <int EPI, int COLS>
__device__ __forceinline__ void store_row(const typename AccType<EPI>::T (&acc)[COLS], const KParams& p, int row,
                                          int col0) {
    if (row >= p.M) return;
    const int N = p.N;
    const bool vec = (N & 7) == 0;
    const int64_t rowoff = static_cast<int64_t>(row) * N;
    float sxr = 0.0f;
    if constexpr (EPI == kEpiPostscaleBf16) sxr = __ldg(p.sx + row);
    const uint16_t* bias16 = reinterpret_cast<const uint16_t*>(p.bias);
#pragma unroll
    for (int j = 0; j < COLS; j += 8) {
        const int col = col0 + j;
        if (col < N) {
            const bool full = vec && (col + 8 <= N);
            if constexpr (EPI == kEpiPostscaleS32 || EPI == kEpiBlockwiseF32) {
                using T = typename AccType<EPI>::T;
                T* out = static_cast<T*>(p.out) + rowoff + col;
                if (full) {
                    uint4 lo, hi;
                    lo.x = *reinterpret_cast<const uint32_t*>(&acc[j + 0]);
                    lo.y = *reinterpret_cast<const uint32_t*>(&acc[j + 1]);
                    lo.z = *reinterpret_cast<const uint32_t*>(&acc[j + 2]);
                    lo.w = *reinterpret_cast<const uint32_t*>(&acc[j + 3]);
                    hi.x = *reinterpret_cast<const uint32_t*>(&acc[j + 4]);
                    hi.y = *reinterpret_cast<const uint32_t*>(&acc[j + 5]);
                    hi.z = *reinterpret_cast<const uint32_t*>(&acc[j + 6]);
                    hi.w = *reinterpret_cast<const uint32_t*>(&acc[j + 7]);
                    reinterpret_cast<uint4*>(out)[0] = lo;
                    reinterpret_cast<uint4*>(out)[1] = hi;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (col + e < N) out[e] = acc[j + e];
                }
            } else {
                float y[8];
                float swc[8];
                float bc[8];
                if (full) {
                    if constexpr (EPI == kEpiPostscaleBf16) {
                        const float4 s0 = __ldg(reinterpret_cast<const float4*>(p.sw + col));
                        const float4 s1 = __ldg(reinterpret_cast<const float4*>(p.sw + col + 4));
                        swc[0] = s0.x; swc[1] = s0.y; swc[2] = s0.z; swc[3] = s0.w;
                        swc[4] = s1.x; swc[5] = s1.y; swc[6] = s1.z; swc[7] = s1.w;
                    }
                    if (p.bias) {
                        const uint4 b = __ldg(reinterpret_cast<const uint4*>(bias16 + col));
                        const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            bc[2 * e] = __uint_as_float(bw[e] << 16);
                            bc[2 * e + 1] = __uint_as_float(bw[e] & 0xFFFF0000u);
                        }
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const bool in = col + e < N;
                        if constexpr (EPI == kEpiPostscaleBf16) swc[e] = in ? __ldg(p.sw + col + e) : 0.0f;
                        if (p.bias) bc[e] = in ? bf16_bits_to_f32(__ldg(bias16 + col + e)) : 0.0f;
                    }
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float v;
                    if constexpr (EPI == kEpiPostscaleBf16)
                        v = __fmul_rn(__fmul_rn(__int2float_rn(acc[j + e]), sxr), swc[e]);
                    else
                        v = acc[j + e];
                    if (p.bias) v = __fadd_rn(v, bc[e]);
                    y[e] = v;
                }
                uint16_t* out = static_cast<uint16_t*>(p.out) + rowoff + col;
                if (full) {
                    uint4 o;
                    o.x = pack_bf16x2(y[0], y[1]);
                    o.y = pack_bf16x2(y[2], y[3]);
                    o.z = pack_bf16x2(y[4], y[5]);
                    o.w = pack_bf16x2(y[6], y[7]);
                    *reinterpret_cast<uint4*>(out) = o;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (col + e < N) {
                            __nv_bfloat16 h = __float2bfloat16_rn(y[e]);
                            out[e] = *reinterpret_cast<uint16_t*>(&h);
                        }
                }
            }
        }
    }
}

// Stage 16 bf16 columns (8 packed words) of each of the warp's 32 rows in a
// 1 KB buffer with the 32-byte swizzle (16-byte chunk index XOR bit 2 of the
// row, which spreads each quarter-warp over 8 bank groups) and store them as
// one 16 x 32 box from one lane.  OUT_BUFS buffers per warp rotate; a buffer
// is rewritten only after the store issued from it has read it.  One buffer
// per warp measured as fast as two and leaves room for a 7th ring stage at
// BN = 224.
// Out-of-range rows and columns are clipped by the TMA unit.
__device__ __forceinline__ void stage_store16(const uint32_t (&o)[8], const CUtensorMap* tmY, int col, int row_base,
                                              uint8_t* stg, int& sbuf, int lane) {
    uint8_t* buf = stg + sbuf * STAGE_OUT_BYTES;
    if (lane == 0) bulk_wait_group_read<OUT_BUFS - 1>();
    __syncwarp();
    const int sw = (lane >> 2) & 1;
    *reinterpret_cast<uint4*>(buf + lane * 32 + 16 * (0 ^ sw)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(buf + lane * 32 + 16 * (1 ^ sw)) = make_uint4(o[4], o[5], o[6], o[7]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(tmY, buf, col, row_base);
        bulk_commit_group();
    }
    sbuf = (sbuf + 1) % OUT_BUFS;
}

// bf16 output of one warp's 32 rows x COLS columns through shared memory and
// TMA stores, 16 columns at a time (stage_store16).
template <int EPI, int COLS>
__device__ __forceinline__ void store_rows_tma(const typename AccType<EPI>::T (&acc)[COLS], const KParams& p,
                                               const CUtensorMap* tmY, int row, int row_base, int col0,
                                               uint8_t* stg, int& sbuf, int lane) {
    float sxr = 0.0f;
    if constexpr (EPI == kEpiPostscaleBf16) sxr = (row < p.M) ? __ldg(p.sx + row) : 0.0f;
    const uint16_t* bias16 = reinterpret_cast<const uint16_t*>(p.bias);
#pragma unroll
    for (int g = 0; g < COLS; g += 16) {
        const int col = col0 + g;
        if (col >= p.N) break;
        float swc[16], bc[16];
        const bool full = col + 16 <= p.N;
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
            if constexpr (EPI == kEpiPostscaleBf16) {
                if (full) {
                    const float4 s4 = __ldg(reinterpret_cast<const float4*>(p.sw + col + e));
                    swc[e] = s4.x; swc[e + 1] = s4.y; swc[e + 2] = s4.z; swc[e + 3] = s4.w;
                } else {
#pragma unroll
                    for (int f = 0; f < 4; ++f) swc[e + f] = (col + e + f < p.N) ? __ldg(p.sw + col + e + f) : 0.0f;
                }
            }
        }
        if (p.bias) {
#pragma unroll
            for (int e = 0; e < 16; e += 8) {
                if (full) {
                    const uint4 b = __ldg(reinterpret_cast<const uint4*>(bias16 + col + e));
                    const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                    for (int f = 0; f < 4; ++f) {
                        bc[e + 2 * f] = __uint_as_float(bw[f] << 16);
                        bc[e + 2 * f + 1] = __uint_as_float(bw[f] & 0xFFFF0000u);
                    }
                } else {
#pragma unroll
                    for (int f = 0; f < 8; ++f)
                        bc[e + f] = (col + e + f < p.N) ? bf16_bits_to_f32(__ldg(bias16 + col + e + f)) : 0.0f;
                }
            }
        }
        uint32_t o[8];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
            float v0, v1;
            if constexpr (EPI == kEpiPostscaleBf16) {
                v0 = __fmul_rn(__fmul_rn(__int2float_rn(acc[g + e]), sxr), swc[e]);
                v1 = __fmul_rn(__fmul_rn(__int2float_rn(acc[g + e + 1]), sxr), swc[e + 1]);
            } else {
                v0 = acc[g + e];
                v1 = acc[g + e + 1];
            }
            if (p.bias) {
                v0 = __fadd_rn(v0, bc[e]);
                v1 = __fadd_rn(v1, bc[e + 1]);
            }
            o[e >> 1] = pack_bf16x2(v0, v1);
        }
        stage_store16(o, tmY, col, row_base, stg, sbuf, lane);
    }
}

// FFN up-projection epilogue, staged.  For each thread's row and its 128
// columns -- exactly one 1x128 block of the down-projection's input --
//   y = bf16(((acc * sx) * sw) + bias)   (the post-scale epilogue),
//   g = bf16(gelu(y))  (gelu.cuh),
//   s = absmax(|g|) / 127, codes = clamp(rne(g / s), -127, 127),
// with the scale written to sg[row][col0 / 128] and the exact bf16 image of
// the codes (the down-projection GEMM's A operand) stored through TMA.
// y leaves the registers at the end of its tile: each thread parks its 256
// bytes in its own row of shared memory (16-byte chunk j at position
// j ^ (lane & 7), which puts the 8 lanes of a quarter-warp on 8 different
// bank groups), and the GELU and quantization then run in eight slices
// spread over the chunk folds of the next tile.
struct GeluStage {
    int row, row_base, col0;  // this thread's staged block
    int slice;                // next slice, 0..7; 8 = nothing pending
    float amax;
    RowScale sc;
};

__device__ __forceinline__ uint4* ychunk(uint8_t* yrow, int j, int lane) {
    return reinterpret_cast<uint4*>(yrow + ((j ^ (lane & 7)) << 4));
}

template <int COLS>
__device__ __forceinline__ void stage_y(const int32_t (&acc)[COLS], const KParams& p, int row, int col0,
                                        uint8_t* yrow, int lane) {
    static_assert(COLS == 128, "one 1x128 block per thread");
    const float sxr = (row < p.M) ? __ldg(p.sx + row) : 0.0f;
    const uint16_t* bias16 = reinterpret_cast<const uint16_t*>(p.bias);
#pragma unroll
    for (int j = 0; j < COLS / 8; ++j) {
        const int col = col0 + 8 * j;
        const float4 s0 = __ldg(reinterpret_cast<const float4*>(p.sw + col));
        const float4 s1 = __ldg(reinterpret_cast<const float4*>(p.sw + col + 4));
        const float swc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
        float bc[8];
        if (p.bias) {
            const uint4 b = __ldg(reinterpret_cast<const uint4*>(bias16 + col));
            const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int f = 0; f < 4; ++f) {
                bc[2 * f] = __uint_as_float(bw[f] << 16);
                bc[2 * f + 1] = __uint_as_float(bw[f] & 0xFFFF0000u);
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            float v0 = __fmul_rn(__fmul_rn(__int2float_rn(acc[8 * j + e]), sxr), swc[e]);
            float v1 = __fmul_rn(__fmul_rn(__int2float_rn(acc[8 * j + e + 1]), sxr), swc[e + 1]);
            if (p.bias) {
                v0 = __fadd_rn(v0, bc[e]);
                v1 = __fadd_rn(v1, bc[e + 1]);
            }
            o[e >> 1] = pack_bf16x2(v0, v1);
        }
        *ychunk(yrow, j, lane) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// One slice of the staged block.  Slices 0-3: g = bf16(gelu(y)) for columns
// 32s .. 32s+31, written back in place, and the running absmax (after slice 3
// the block scale is known and stored).  Slices 4-7: the codes of columns
// 32(s-4) .. +31 as their bf16 image, out through two 16 x 32 TMA boxes.
__device__ __forceinline__ void gelu_slice(GeluStage& gs, const KParams& p, const CUtensorMap* tmY, uint8_t* yrow,
                                           uint8_t* stg, int& sbuf, int lane) {
    const int s = gs.slice++;
    if (s < 4) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4* ptr = ychunk(yrow, 4 * s + q, lane);
            const uint4 v = *ptr;
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t g[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                g[i] = gelu_bf16x2(bf16_lo(w[i]), bf16_hi(w[i]));
                gs.amax = fmaxf(gs.amax, fmaxf(fabsf(bf16_lo(g[i])), fabsf(bf16_hi(g[i]))));
            }
            *ptr = make_uint4(g[0], g[1], g[2], g[3]);
        }
        if (s == 3) {
            gs.sc = make_scale_div(gs.amax);
            if (gs.row < p.M) p.sg[static_cast<int64_t>(gs.row) * (p.N >> 7) + (gs.col0 >> 7)] = gs.sc.s;
        }
    } else {
        const int b = s - 4;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int j0 = 4 * b + 2 * h;
            const uint4 c0 = quant_chunk_img(*ychunk(yrow, j0, lane), gs.sc);
            const uint4 c1 = quant_chunk_img(*ychunk(yrow, j0 + 1, lane), gs.sc);
            const uint32_t o[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            stage_store16(o, tmY, gs.col0 + 32 * b + 16 * h, gs.row_base, stg, sbuf, lane);
        }
    }
}

// Split K (swapped operands only): this unit's exact int32 partial sums, for
// output column n = kernel row and COLS tokens, into slice `split` of the
// partial buffer [k_split][tokens][N]; lanes write consecutive n.
template <int COLS>
__device__ __forceinline__ void store_partial(const int32_t (&acc)[COLS], const KParams& p, int n_base, int tok0,
                                              int split, int lane) {
    const int n = n_base + lane;
    const int Nout = p.M, Mtok = p.N;
    if (n >= Nout) return;
    int32_t* dst = p.partial + (static_cast<int64_t>(split) * Mtok + tok0) * Nout + n;
#pragma unroll
    for (int e = 0; e < COLS; ++e)
        if (tok0 + e < Mtok) dst[static_cast<int64_t>(e) * Nout] = acc[e];
}

// Swapped operands (few tokens): the kernel's rows are weight rows n and its
// columns are tokens m, so this thread holds output column n for COLS tokens.
// y = ((float(acc) * sx[m]) * sw[n]) + bias[n], the same operations in the
// same order as the unswapped epilogue.  bf16 output goes through shared
// memory as [16 tokens x 32 columns] boxes (one 2-byte value per lane per
// token row) and a TMA store into Y[m][n]; the int32 export and rows of N not
// a multiple of 8 use direct stores.
template <int EPI, int COLS>
__device__ __forceinline__ void store_swapped(const int32_t (&acc)[COLS], const KParams& p, const CUtensorMap* tmY,
                                              int n_base, int tok0, uint8_t* stg, int& sbuf, int lane) {
    const int n = n_base + lane;       // output column (kernel row)
    const int Nout = p.M, Mtok = p.N;  // kernel dims: rows = weights, columns = tokens
    if constexpr (EPI == kEpiPostscaleS32) {
        if (n < Nout) {
#pragma unroll
            for (int e = 0; e < COLS; ++e)
                if (tok0 + e < Mtok) static_cast<int32_t*>(p.out)[static_cast<int64_t>(tok0 + e) * Nout + n] = acc[e];
        }
        return;
    } else {
        const float swn = (n < Nout) ? __ldg(p.sw + n) : 0.0f;
        const float bn = (p.bias && n < Nout) ? bf16_bits_to_f32(__ldg(reinterpret_cast<const uint16_t*>(p.bias) + n))
                                              : 0.0f;
#pragma unroll
        for (int g = 0; g < COLS; g += 16) {
            const int t0 = tok0 + g;
            if (t0 >= Mtok) break;
            float sxt[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) sxt[e] = (t0 + e < Mtok) ? __ldg(p.sx + t0 + e) : 0.0f;
            uint16_t y[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                float v = __fmul_rn(__fmul_rn(__int2float_rn(acc[g + e]), sxt[e]), swn);
                if (p.bias) v = __fadd_rn(v, bn);
                __nv_bfloat16 h = __float2bfloat16_rn(v);
                y[e] = *reinterpret_cast<uint16_t*>(&h);
            }
            if (p.tma_store) {
                uint8_t* buf = stg + sbuf * STAGE_OUT_BYTES;
                if (lane == 0) bulk_wait_group_read<OUT_BUFS - 1>();
                __syncwarp();
#pragma unroll
                for (int e = 0; e < 16; ++e) *reinterpret_cast<uint16_t*>(buf + e * 64 + lane * 2) = y[e];
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(tmY, buf, n_base, t0);
                    bulk_commit_group();
                }
                sbuf = (sbuf + 1) % OUT_BUFS;
            } else if (n < Nout) {
                uint16_t* out = static_cast<uint16_t*>(p.out);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (t0 + e < Mtok) out[static_cast<int64_t>(t0 + e) * Nout + n] = y[e];
            }
        }
    }
}

template <int EPI, int BN, bool SWAP>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmY, const KParams p) {
    grid_launch_dependents();
    using C = Cfg<BN, EPI == kEpiGeluQuant ? YSTAGE_BYTES : 0u>;
    constexpr int STAGES = C::STAGES;
    constexpr int HALF = C::HALF;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_BYTES;
    uint8_t* staging = sB + STAGES * C::B_BYTES;  // 1 KB aligned
    uint8_t* ystage = staging + STAGING_BYTES;  // kEpiGeluQuant only (1 KB aligned)
    uint64_t* full = reinterpret_cast<uint64_t*>(ystage + (EPI == kEpiGeluQuant ? YSTAGE_BYTES : 0u));
    uint64_t* empty = full + STAGES;
    uint64_t* acc_full = empty + STAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* mma_drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: leader (issues the MMAs), 1: peer
    const bool leader = rank == 0;
    const int cluster = static_cast<int>(cluster_id_x());
    const int nclusters = static_cast<int>(nclusters_x());

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);   // leader only: its arrive + both CTAs' bytes
            mbar_init(&empty[s], 1);  // both: the leader's multicast commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);               // both: multicast commit
            mbar_init(&acc_empty[b], 2 * EPI_WARPS);  // leader only: every epilogue warp of the pair
        }
        mbar_init(mma_drain, 1);
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer's barriers are initialized before anyone signals them
    tc_fence_after();
    // Everything above overlaps the tail of the kernel that wrote the
    // operands and scales (programmatic dependent launch); nothing below
    // reads global memory before that kernel has completed -- except the
    // producer's first fills of a settled operand (a weight image packed
    // before the previous kernel started), which it issues before its own
    // dependency wait.
    if (warp != 0) grid_dependency_wait();
    const uint32_t tmem_base = *tmem_slot;
    if (warp < EPI_WARP0) {
      regs_dec<REGS_LOW>();
      if (warp == 0) {
        // ------------------------------------------------------------ producer (both CTAs)
        const bool elected = elect_one_sync();
        // Stages of the first unit whose settled operand went out before the
        // dependency wait (the ring's first fills need no empty wait).
        int pre = 0;
        if (elected && (p.a_settled || p.b_settled) && cluster < p.num_tiles) {
            const Unit w = unit_coords(cluster, p);
            pre = min(STAGES, w.ks1 - w.ks0);
            const int a_row = w.mb * TILE_M + static_cast<int>(rank) * BM;
            const int b_row = w.nb * BN + static_cast<int>(rank) * HALF;
            for (int i = 0; i < pre; ++i) {
                if (leader) mbar_arrive_expect_tx(&full[i], 2 * C::STAGE_BYTES);
                const uint32_t bar = map_to_rank(smem_u32(&full[i]), 0);
                if (p.a_settled) tma_load_2d_pair(sA + i * A_BYTES, &tmA, bar, (w.ks0 + i) * BK, a_row);
                else tma_load_2d_pair(sB + i * C::B_BYTES, &tmB, bar, (w.ks0 + i) * BK, b_row);
            }
        }
        grid_dependency_wait();
        if (elected) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_phase = 0;
            bool ok = true;
            for (int u = cluster; ok && u < p.num_tiles; u += nclusters) {
                const Unit w = unit_coords(u, p);
                const int a_row = w.mb * TILE_M + static_cast<int>(rank) * BM;
                const int b_row = w.nb * BN + static_cast<int>(rank) * HALF;
                for (int ks = w.ks0; ks < w.ks1; ++ks) {
                    const uint32_t bar = map_to_rank(smem_u32(&full[stage]), 0);
                    if (u == cluster && ks - w.ks0 < pre) {
                        // first fill, settled half already in flight
                        if (p.a_settled) tma_load_2d_pair(sB + stage * C::B_BYTES, &tmB, bar, ks * BK, b_row);
                        else tma_load_2d_pair(sA + stage * A_BYTES, &tmA, bar, ks * BK, a_row);
                    } else {
                        if (!mbar_wait(&empty[stage], phase ^ 1u, kSiteProducerEmpty)) {
                            ok = false;
                            break;
                        }
                        if (leader) mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE_BYTES);
                        tma_load_2d_pair(sA + stage * A_BYTES, &tmA, bar, ks * BK, a_row);
                        tma_load_2d_pair(sB + stage * C::B_BYTES, &tmB, bar, ks * BK, b_row);
                    }
                    armed |= 1u << stage;
                    armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // The MMAs that read each stage's last fill have completed (so its
            // copies landed) before this CTA's shared memory is released.
            for (int s = 0; s < STAGES; ++s)
                if (armed & (1u << s)) mbar_wait(&empty[s], (armed_phase >> s) & 1u, kSiteProducerDrain);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader only)
        if (leader && elect_one_sync()) {
            int stage = 0;
            uint32_t phase = 0;
            int buf = 0;
            uint32_t buf_phase = 0;
            bool ok = true;
            // Shared-memory descriptors of stage 0; a stage's descriptors differ
            // only in the start address field (bits 0-13, address >> 4), which
            // stays below 2^14 for any stage, so each stage's low words are a
            // running sum and each K step adds 32 bytes (2) to them.
            const uint64_t dA0 = smem_desc_kmajor_sw128(smem_u32(sA));
            const uint64_t dB0 = smem_desc_kmajor_sw128(smem_u32(sB));
            const uint32_t hiA = static_cast<uint32_t>(dA0 >> 32), hiB = static_cast<uint32_t>(dB0 >> 32);
            uint32_t loA = static_cast<uint32_t>(dA0), loB = static_cast<uint32_t>(dB0);
            for (int u = cluster; ok && u < p.num_tiles; u += nclusters) {
                const Unit w = unit_coords(u, p);
                const int nchunks = (w.ks1 - w.ks0 + p.chunk_stages - 1) / p.chunk_stages;
                for (int c = 0; ok && c < nchunks; ++c) {
                    if (!mbar_wait(&acc_empty[buf], buf_phase ^ 1u, kSiteMmaAccEmpty)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
                    const int s0 = w.ks0 + c * p.chunk_stages;
                    const int s1 = min(w.ks1, s0 + p.chunk_stages);
                    for (int ks = s0; ks < s1; ++ks) {
                        if (!mbar_wait(&full[stage], phase, kSiteMmaFull)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k) {
                            const uint64_t da = (static_cast<uint64_t>(hiA) << 32) | (loA + 2u * k);
                            const uint64_t db = (static_cast<uint64_t>(hiB) << 32) | (loB + 2u * k);
                            mma_bf16_ss_pair(d_tmem, da, db, C::IDESC, (ks > s0 || k > 0) ? 1u : 0u);
                        }
                        mma_commit_pair_multicast(&empty[stage], 0x3);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                            loA = static_cast<uint32_t>(dA0);
                            loB = static_cast<uint32_t>(dB0);
                        } else {
                            loA += A_BYTES >> 4;
                            loB += C::B_BYTES >> 4;
                        }
                    }
                    if (!ok) break;
                    mma_commit_pair_multicast(&acc_full[buf], 0x3);
                    buf ^= 1;
                    if (buf == 0) buf_phase ^= 1u;
                }
            }
            // Every MMA issued has completed before TMEM is freed.
            mma_commit_pair(mma_drain);
            mbar_wait(mma_drain, 0, kSiteMmaDrain);
        }
      }
    } else {
        regs_inc<REGS_HIGH>();
        // ------------------------------------------------------------ epilogue (both CTAs)
        constexpr bool kBlock = (EPI == kEpiBlockwiseBf16 || EPI == kEpiBlockwiseF32);
        static_assert(!kBlock || HALF == 128, "blockwise needs each warp's columns inside one 128-wide block");
        static_assert(!(kBlock && SWAP), "swapped operands are for the post-scale GEMM only");
        using T = typename AccType<EPI>::T;
        constexpr int LDW = C::LDW;
        constexpr int GROUPS = C::GROUPS;
        const int quarter = warp & 3;                  // TMEM lanes this warp may access
        const int half = (warp - EPI_WARP0) >> 2;      // which column half of the tile
        const uint32_t leader_acc_empty0 = map_to_rank(smem_u32(&acc_empty[0]), 0);
        constexpr bool kBf16Out = (EPI == kEpiPostscaleBf16 || EPI == kEpiBlockwiseBf16);
        uint8_t* stg = staging + (warp - EPI_WARP0) * OUT_BUFS * STAGE_OUT_BYTES;
        int sbuf = 0;
        int buf = 0;
        uint32_t buf_phase = 0;
        bool ok = true;
        if constexpr (EPI == kEpiGeluQuant) {
            // Tile t's y is staged at the end of t; its eight GELU /
            // quantization slices run ceil(8 / chunks) at a time after the
            // chunk folds of tile t+1 (the rest at its last chunk, or after
            // the last tile), so the MMA never waits behind a whole tile's
            // GELU for a free accumulator buffer.
            uint8_t* yrow = ystage + (warp - EPI_WARP0) * (32 * 256) + lane * 256;
            GeluStage gs;
            gs.row = gs.row_base = gs.col0 = 0;
            gs.slice = 8;
            gs.amax = 0.0f;
            gs.sc = make_scale_div(0.0f);
            for (int u = cluster; ok; u += nclusters) {
                const bool real = u < p.num_tiles;
                if (!real && gs.slice >= 8) break;
                int nchunks = 0, row_base = 0, col0 = 0;
                if (real) {
                    const Unit w = unit_coords(u, p);
                    nchunks = (w.ks1 - w.ks0 + p.chunk_stages - 1) / p.chunk_stages;
                    row_base = w.mb * TILE_M + static_cast<int>(rank) * BM + quarter * 32;
                    col0 = w.nb * BN + half * HALF;
                }
                const int passes = nchunks > 0 ? nchunks : 1;
                const int per = (8 + passes - 1) / passes;
                int32_t acc[HALF];
#pragma unroll
                for (int e = 0; e < HALF; ++e) acc[e] = 0;
                for (int c = 0; c < passes; ++c) {
                    if (real) {
                        if (!mbar_wait(&acc_full[buf], buf_phase, kSiteEpiAccFull)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                               static_cast<uint32_t>(buf * BN + half * HALF);
                        uint32_t ra[LDW], rb[LDW];
                        tmem_ld_cols<LDW>(taddr, ra);
                        tmem_wait_cols(ra);
#pragma unroll
                        for (int j = 0; j < GROUPS; ++j) {
                            uint32_t(&cur)[LDW] = (j & 1) ? rb : ra;
                            uint32_t(&nxt)[LDW] = (j & 1) ? ra : rb;
                            if (j + 1 < GROUPS) tmem_ld_cols<LDW>(taddr + (j + 1) * LDW, nxt);
#pragma unroll
                            for (int e = 0; e < LDW; ++e) acc[j * LDW + e] += __float2int_rz(__uint_as_float(cur[e]));
                            if (j + 1 < GROUPS) tmem_wait_cols(nxt);
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive_cluster_relaxed(leader_acc_empty0 + static_cast<uint32_t>(buf) * 8u);
                        buf ^= 1;
                        if (buf == 0) buf_phase ^= 1u;
                    }
                    int todo = (c + 1 == passes) ? 8 : per;
                    while (gs.slice < 8 && todo-- > 0) gelu_slice(gs, p, &tmY, yrow, stg, sbuf, lane);
                }
                if (!ok || !real) break;
                if (col0 < p.N) {
                    stage_y<HALF>(acc, p, row_base + lane, col0, yrow, lane);
                    gs.row = row_base + lane;
                    gs.row_base = row_base;
                    gs.col0 = col0;
                    gs.slice = 0;
                    gs.amax = 0.0f;
                }
            }
        } else {
        for (int u = cluster; ok && u < p.num_tiles; u += nclusters) {
            const Unit w = unit_coords(u, p);
            const int mb = w.mb, nb = w.nb;
            const int nchunks = (w.ks1 - w.ks0 + p.chunk_stages - 1) / p.chunk_stages;
            const int row_base = mb * TILE_M + static_cast<int>(rank) * BM + quarter * 32;
            const int row = row_base + lane;
            const int col0 = nb * BN + half * HALF;
            // post-scale: int32 running sums; blockwise: fp32 accumulators
            T acc[HALF];
#pragma unroll
            for (int e = 0; e < HALF; ++e) acc[e] = T(0);
            // blockwise: the per-block scales of chunk c are loaded SCALE_PREFETCH
            // chunks ahead (a row's scales are 4-byte loads scattered over 32
            // rows per warp; one chunk ahead left their latency exposed)
            const float* sx_row = p.sx + static_cast<int64_t>(row < p.M ? row : 0) * p.kb_count;
            const float* sw_row = p.sw + static_cast<int64_t>(col0 < p.N ? (col0 >> 7) : 0) * p.kb_count;
            float sxq[SCALE_PREFETCH], swq[SCALE_PREFETCH];
            if constexpr (kBlock) {
#pragma unroll
                for (int i = 0; i < SCALE_PREFETCH; ++i) {
                    sxq[i] = (row < p.M && i < nchunks) ? __ldg(sx_row + i) : 0.0f;
                    swq[i] = (col0 < p.N && i < nchunks) ? __ldg(sw_row + i) : 0.0f;
                }
            }
            for (int c = 0; c < nchunks; ++c) {
                float sxv = 0.0f, swv = 0.0f;
                if constexpr (kBlock) {
                    sxv = sxq[0];
                    swv = swq[0];
#pragma unroll
                    for (int i = 0; i + 1 < SCALE_PREFETCH; ++i) {
                        sxq[i] = sxq[i + 1];
                        swq[i] = swq[i + 1];
                    }
                    const int cn = c + SCALE_PREFETCH;
                    sxq[SCALE_PREFETCH - 1] = (row < p.M && cn < nchunks) ? __ldg(sx_row + cn) : 0.0f;
                    swq[SCALE_PREFETCH - 1] = (col0 < p.N && cn < nchunks) ? __ldg(sw_row + cn) : 0.0f;
                }
                if (!mbar_wait(&acc_full[buf], buf_phase, kSiteEpiAccFull)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                       static_cast<uint32_t>(buf * BN + half * HALF);
                // GROUPS groups of LDW columns; the load of group j+1 is in
                // flight while group j is folded.
                uint32_t ra[LDW], rb[LDW];
                tmem_ld_cols<LDW>(taddr, ra);
                tmem_wait_cols(ra);
#pragma unroll
                for (int j = 0; j < GROUPS; ++j) {
                    uint32_t(&cur)[LDW] = (j & 1) ? rb : ra;
                    uint32_t(&nxt)[LDW] = (j & 1) ? ra : rb;
                    if (j + 1 < GROUPS) tmem_ld_cols<LDW>(taddr + (j + 1) * LDW, nxt);
                    if constexpr (kBlock) {
                        // t = (P * sx) * sw; acc = acc + t, each rounded on its own.  The two
                        // products of a column pair run on the packed fp32 pipe (a product
                        // feeding a product, nothing to contract); the additions stay scalar
                        // with explicit rounding (chained packed multiply-adds get contracted).
                        const uint64_t sx2 = f2_pack(sxv, sxv), sw2 = f2_pack(swv, swv);
#pragma unroll
                        for (int e = 0; e < LDW; e += 2) {
                            float t0, t1;
                            f2_unpack(f2_mul(f2_mul(f2_pack(__uint_as_float(cur[e]), __uint_as_float(cur[e + 1])),
                                                    sx2),
                                             sw2),
                                      t0, t1);
                            acc[j * LDW + e] = __fadd_rn(acc[j * LDW + e], t0);
                            acc[j * LDW + e + 1] = __fadd_rn(acc[j * LDW + e + 1], t1);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < LDW; ++e) acc[j * LDW + e] += __float2int_rz(__uint_as_float(cur[e]));
                    }
                    if (j + 1 < GROUPS) tmem_wait_cols(nxt);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_relaxed(leader_acc_empty0 + static_cast<uint32_t>(buf) * 8u);
                buf ^= 1;
                if (buf == 0) buf_phase ^= 1u;
            }
            if (!ok) break;
            if constexpr (SWAP) {
                if constexpr (!kBlock) {
                    if (p.k_split > 1)
                        store_partial<HALF>(acc, p, row_base, col0, w.split, lane);
                    else
                        store_swapped<EPI, HALF>(acc, p, &tmY, row_base, col0, stg, sbuf, lane);
                }
            } else if (kBf16Out && p.tma_store) {
                store_rows_tma<EPI, HALF>(acc, p, &tmY, row, row_base, col0, stg, sbuf, lane);
            } else {
                store_row<EPI, HALF>(acc, p, row, col0);
            }
        }
        }  // EPI != kEpiGeluQuant
        if (lane == 0) bulk_wait_group_all();  // this warp's output stores have completed
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // neither CTA leaves while the pair may still touch its barriers or smem
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// Split K, last step: Y[m][n] from the sum of the k_split int32 partials of
// output (m, n) -- integer additions, exact in any order -- then the
// post-scale epilogue in the unsplit kernel's operation order.  Launched as a
// programmatic dependent of the GEMM; one thread per output, lanes along n.
template <int EPI>
__global__ void __launch_bounds__(256) splitk_finalize_kernel(const int32_t* __restrict__ partial, int k_split,
                                                              int M, int N, const float* __restrict__ sx,
                                                              const float* __restrict__ sw,
                                                              const __nv_bfloat16* __restrict__ bias,
                                                              void* __restrict__ out) {
    grid_dependency_wait();
    const int64_t total = static_cast<int64_t>(M) * N;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        int32_t acc = 0;
        for (int s = 0; s < k_split; ++s) acc += __ldcs(partial + s * total + i);
        if constexpr (EPI == kEpiPostscaleS32) {
            static_cast<int32_t*>(out)[i] = acc;
        } else {
            const int m = static_cast<int>(i / N);
            const int n = static_cast<int>(i - static_cast<int64_t>(m) * N);
            float v = __fmul_rn(__fmul_rn(__int2float_rn(acc), __ldg(sx + m)), __ldg(sw + n));
            if (bias) v = __fadd_rn(v, bf16_bits_to_f32(__ldg(reinterpret_cast<const uint16_t*>(bias) + n)));
            static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
        }
    }
}

CUresult make_map(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* map, const void* base, int64_t inner,
                  int64_t rows, uint32_t box_inner, uint32_t box_rows) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * 2};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Per device: whether each kernel instance has its shared-memory attribute set,
// and how many CTA pairs of the GEMM kernel fit at once.
struct DeviceLaunchInfo {
    bool configured[32];
    int max_clusters;
};
DeviceLaunchInfo g_launch_info[64];

template <int EPI, int BN, bool SWAP>
constexpr int instance_id() {
    return (EPI == kEpiPostscaleBf16 ? 0 : EPI == kEpiPostscaleS32 ? 8 : EPI == kEpiBlockwiseBf16 ? 16
            : EPI == kEpiBlockwiseF32 ? 17 : 18) +
           (SWAP ? 4 : 0) +
           (BN == 256 ? 0 : BN == 224 ? 1 : BN == 192 ? 2 : BN == 128 ? 1 : BN == 64 ? 2 : 3);
}

// Launch one kernel instance.  Ab / Bb are the operand images of the kernel's
// rows and columns; p.M / p.N are the kernel's dimensions (with SWAP the rows
// are weight rows and the columns tokens, and Y is written transposed).
template <int EPI, int BN, bool SWAP>
cudaError_t launch_one(const void* Ab, const void* Bb, PFN_cuTensorMapEncodeTiled_v12000 encode, KParams p,
                       int num_sms, cudaStream_t st, char* detail, size_t n) {
    using C = Cfg<BN, EPI == kEpiGeluQuant ? YSTAGE_BYTES : 0u>;
    CUtensorMap tmA, tmB;
    CUresult r = make_map(encode, &tmA, Ab, p.K, p.M, BK, BM);
    if (r != CUDA_SUCCESS) {
        snprintf(detail, n, "cuTensorMapEncodeTiled(A: %d x %d) returned %d", p.M, p.K, (int)r);
        return cudaErrorInvalidValue;
    }
    r = make_map(encode, &tmB, Bb, p.K, p.N, BK, C::HALF);
    if (r != CUDA_SUCCESS) {
        snprintf(detail, n, "cuTensorMapEncodeTiled(B: %d x %d) returned %d", p.N, p.K, (int)r);
        return cudaErrorInvalidValue;
    }
    CUtensorMap tmY = tmB;  // placeholder when the output is not written through TMA
    constexpr bool kBf16Out = (EPI == kEpiPostscaleBf16 || EPI == kEpiBlockwiseBf16 || EPI == kEpiGeluQuant);
    const int y_cols = SWAP ? p.M : p.N;  // Y is [tokens, output columns]
    const int y_rows = SWAP ? p.N : p.M;
    p.tma_store = (kBf16Out && (y_cols % 8) == 0) ? 1 : 0;
    if (p.tma_store) {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(y_cols), static_cast<cuuint64_t>(y_rows)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(y_cols) * 2};
        cuuint32_t box[2] = {SWAP ? 32u : 16u, SWAP ? 16u : 32u};
        cuuint32_t estr[2] = {1, 1};
        r = encode(&tmY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.out, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, SWAP ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_32B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            snprintf(detail, n, "cuTensorMapEncodeTiled(Y: %d x %d) returned %d", p.M, p.N, (int)r);
            return cudaErrorInvalidValue;
        }
    }
    p.num_m = (p.M + TILE_M - 1) / TILE_M;
    p.num_n = (p.N + BN - 1) / BN;
    p.num_tiles = p.num_m * p.num_n * p.k_split;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    DeviceLaunchInfo& info = g_launch_info[dev];
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;  // the occupancy query below takes the cluster shape only
    constexpr int id = instance_id<EPI, BN, SWAP>();
    if (!info.configured[id]) {
        e = cudaFuncSetAttribute(gemm_kernel<EPI, BN, SWAP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(C::SMEM));
        if (e != cudaSuccess) return e;
        if (info.max_clusters == 0) {
            cfg.gridDim = dim3(2 * (num_sms / 2));
            int nc = 0;
            e = cudaOccupancyMaxActiveClusters(&nc, gemm_kernel<EPI, BN, SWAP>, &cfg);
            if (e != cudaSuccess) return e;
            if (nc < 1) {
                snprintf(detail, n, "no CTA pair of the GEMM kernel fits on this device");
                return cudaErrorInvalidConfiguration;
            }
            info.max_clusters = nc;
        }
        info.configured[id] = true;
    }
    const int clusters = p.num_tiles < info.max_clusters ? p.num_tiles : info.max_clusters;
    cfg.gridDim = dim3(2 * clusters);
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gemm_kernel<EPI, BN, SWAP>, tmA, tmB, tmY, p);
}

// Tile width for the post-scale GEMM: the candidate minimizing
// waves x (BN + 16), i.e. whole waves of CTA pairs times the per-tile MMA
// time plus a fixed per-tile cost.
int choose_bn(int64_t M, int64_t N, int clusters) {
    const int cand[4] = {256, 224, 192, 160};
    const int64_t mt = (M + TILE_M - 1) / TILE_M;
    int best = 256;
    int64_t best_cost = -1;
    for (int bn : cand) {
        const int64_t tiles = mt * ((N + bn - 1) / bn);
        const int64_t waves = (tiles + clusters - 1) / clusters;
        const int64_t cost = waves * (bn + 16);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = bn;
        }
    }
    return best;
}

template <int EPI>
cudaError_t launch_bn(int bn, const void* Ab, const void* Bb, PFN_cuTensorMapEncodeTiled_v12000 encode,
                      const KParams& p, int num_sms, cudaStream_t st, char* detail, size_t n) {
    switch (bn) {
        case 224: return launch_one<EPI, 224, false>(Ab, Bb, encode, p, num_sms, st, detail, n);
        case 192: return launch_one<EPI, 192, false>(Ab, Bb, encode, p, num_sms, st, detail, n);
        case 160: return launch_one<EPI, 160, false>(Ab, Bb, encode, p, num_sms, st, detail, n);
        default: return launch_one<EPI, 256, false>(Ab, Bb, encode, p, num_sms, st, detail, n);
    }
}

// Few tokens (M <= 256): weights take the 256-row side of the CTA-pair MMA and
// the tokens its N side (the narrowest of 32 / 64 / 128 / 256 that holds them).
template <int EPI>
cudaError_t launch_swapped(const void* Ximg, const void* Wimg, PFN_cuTensorMapEncodeTiled_v12000 encode, KParams p,
                           int num_sms, cudaStream_t st, char* detail, size_t n) {
    const int tokens = p.M;
    p.M = p.N;  // kernel rows: weight rows
    p.N = tokens;
    const int settled = p.a_settled;
    p.a_settled = p.b_settled;
    p.b_settled = settled;
    if (tokens <= 32) return launch_one<EPI, 32, true>(Wimg, Ximg, encode, p, num_sms, st, detail, n);
    if (tokens <= 64) return launch_one<EPI, 64, true>(Wimg, Ximg, encode, p, num_sms, st, detail, n);
    if (tokens <= 128) return launch_one<EPI, 128, true>(Wimg, Ximg, encode, p, num_sms, st, detail, n);
    return launch_one<EPI, 256, true>(Wimg, Ximg, encode, p, num_sms, st, detail, n);
}

template <int EPI>
cudaError_t launch_finalize(const KParams& p, const GemmArgs& a, int num_sms, cudaStream_t st) {
    const int64_t total = a.M * a.N;
    int64_t grid = (total + 255) / 256;
    if (grid > static_cast<int64_t>(num_sms) * 8) grid = static_cast<int64_t>(num_sms) * 8;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, splitk_finalize_kernel<EPI>, static_cast<const int32_t*>(p.partial), p.k_split,
                              static_cast<int>(a.M), static_cast<int>(a.N), a.sx, a.sw,
                              static_cast<const __nv_bfloat16*>(a.bias), a.out);
}

}  // namespace

bool gemm_takes_int8(int epilogue, int64_t M) {
    return (epilogue == kEpiPostscaleBf16 || epilogue == kEpiPostscaleS32) && M > 0 && M <= kInt8MaxTokens;
}

int splitk_plan(bool blockwise, int64_t M, int64_t N, int64_t K, int* split_stages) {
    const int64_t k_stages = (K + BK - 1) / BK;
    if (split_stages) *split_stages = static_cast<int>(k_stages);
    if (blockwise || M <= 0 || M > kSwapMaxTokens || N <= 0 || K <= 0) return 1;
    const int64_t tiles = (N + TILE_M - 1) / TILE_M;
    int64_t s = kSplitTargetUnits / tiles;
    if (s > k_stages / kSplitMinStages) s = k_stages / kSplitMinStages;
    if (s > kSplitMax) s = kSplitMax;
    if (s < 2) return 1;
    const int64_t per = (k_stages + s - 1) / s;  // stages per split; no split is left empty
    if (split_stages) *split_stages = static_cast<int>(per);
    return static_cast<int>((k_stages + per - 1) / per);
}

size_t splitk_partial_bytes(int64_t M, int64_t N, int64_t K) {
    const int s = splitk_plan(false, M, N, K, nullptr);
    return s > 1 ? static_cast<size_t>(s) * static_cast<size_t>(M) * static_cast<size_t>(N) * 4 : 0;
}

cudaError_t launch_gemm(int epilogue, const void* Ab, const void* Bb, const GemmArgs& a, int num_sms,
                        void* encode_fn, cudaStream_t st, char* detail, size_t n) {
    if (n) detail[0] = 0;
    if (a.int8_operands && !gemm_takes_int8(epilogue, a.M)) {
        snprintf(detail, n, "int8 operands are taken only by the few-token post-scale GEMM");
        return cudaErrorInvalidValue;
    }
    if (a.int8_operands) return launch_gemm_s8(epilogue, Ab, Bb, a, num_sms, encode_fn, st, detail, n);
    auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(encode_fn);
    KParams p;
    p.sx = a.sx;
    p.sw = a.sw;
    p.bias = static_cast<const __nv_bfloat16*>(a.bias);
    p.out = a.out;
    p.sg = a.sg;
    p.a_settled = 0;
    p.b_settled = a.weights_settled ? 1 : 0;  // B holds the weights (swapped launches exchange the flags)
    p.group_m = (epilogue == kEpiBlockwiseBf16 || epilogue == kEpiBlockwiseF32) ? GROUP_M_BLOCKWISE
                                                                                : GROUP_M_POSTSCALE;
    p.M = static_cast<int>(a.M);
    p.N = static_cast<int>(a.N);
    p.K = static_cast<int>(a.K);
    p.k_stages = static_cast<int>((a.K + BK - 1) / BK);
    const bool blockwise = epilogue == kEpiBlockwiseBf16 || epilogue == kEpiBlockwiseF32;
    p.chunk_stages = blockwise ? BLOCK_CHUNK_STAGES : POSTSCALE_CHUNK_STAGES;
    p.kb_count = static_cast<int>(a.K / 128);
    const bool swap = !blockwise && epilogue != kEpiGeluQuant && a.M <= kSwapMaxTokens;
    p.k_split = 1;
    p.split_stages = p.k_stages;
    p.partial = nullptr;
    if (swap) {
        int per = 0;
        const int ks = splitk_plan(false, a.M, a.N, a.K, &per);
        if (ks > 1) {
            if (!a.partial) {
                snprintf(detail, n, "split-K GEMM without a partial-sum buffer");
                return cudaErrorInvalidValue;
            }
            p.k_split = ks;
            p.split_stages = per;
            p.partial = a.partial;
        }
    }
    const int bn = blockwise ? 256 : choose_bn(a.M, a.N, num_sms / 2);
    cudaError_t e;
    switch (epilogue) {
        case kEpiPostscaleBf16:
            e = swap ? launch_swapped<kEpiPostscaleBf16>(Ab, Bb, encode, p, num_sms, st, detail, n)
                     : launch_bn<kEpiPostscaleBf16>(bn, Ab, Bb, encode, p, num_sms, st, detail, n);
            break;
        case kEpiPostscaleS32:
            e = swap ? launch_swapped<kEpiPostscaleS32>(Ab, Bb, encode, p, num_sms, st, detail, n)
                     : launch_bn<kEpiPostscaleS32>(bn, Ab, Bb, encode, p, num_sms, st, detail, n);
            break;
        case kEpiBlockwiseBf16:
            e = launch_one<kEpiBlockwiseBf16, 256, false>(Ab, Bb, encode, p, num_sms, st, detail, n);
            break;
        case kEpiBlockwiseF32:
            e = launch_one<kEpiBlockwiseF32, 256, false>(Ab, Bb, encode, p, num_sms, st, detail, n);
            break;
        case kEpiGeluQuant:
            // 256-wide tiles: each epilogue thread holds one whole 1x128 block
            e = launch_one<kEpiGeluQuant, 256, false>(Ab, Bb, encode, p, num_sms, st, detail, n);
            break;
        default: e = cudaErrorInvalidValue;
    }
    if (e == cudaSuccess && p.k_split > 1)
        e = epilogue == kEpiPostscaleS32 ? launch_finalize<kEpiPostscaleS32>(p, a, num_sms, st)
                                         : launch_finalize<kEpiPostscaleBf16>(p, a, num_sms, st);
    if (e != cudaSuccess && n && detail[0] == 0)
        snprintf(detail, n, "GEMM launch (%d threads, clusters of 2, tile width %d): %s", THREADS, bn,
                 cudaGetErrorString(e));
    return e;
}

namespace {

constexpr int kSiteProbe = 30;

// Failure-detection probe: one thread waits on an mbarrier that nothing
// arrives on.  The bounded wait runs out, records the timeout in this
// translation unit's device error word, and the kernel returns normally.
__global__ void wait_timeout_probe_kernel() {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, kSiteProbe);
}

}  // namespace

cudaError_t launch_wait_timeout_probe(cudaStream_t st) {
    wait_timeout_probe_kernel<<<1, 32, 0, st>>>();
    return cudaGetLastError();
}

cudaError_t gemm_read_device_error(unsigned int* code) {
    unsigned int v = 0, z = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof v);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbol(g_device_error, &z, sizeof z);
    *code = v;
    return e;
}

}  // namespace w8a8
