// Few-token post-scale W8A8 GEMM on the int8 codes themselves (5..288
// tokens): the weight codes stream once from HBM and are widened into tensor
// memory, the tokens arrive as an fp16 image of their codes, and the exact
// integer product runs on the fp16 tcgen05 pipe.  launch_gemm (gemm.cu)
// routes int8-operand calls here: up to 96 tokens to gemm_s8_kernel, beyond
// that to gemm_s8w_kernel (whose 160-token tile also beats a 128-token tile
// of the first kernel from 97 tokens on).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdio>

#include "kernels.h"
#include "ptx.cuh"

namespace w8a8 {
namespace {

constexpr int BM = 128;                       // weight rows per CTA (M of the MMA)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t MAX_DYN_SMEM = 232448;     // 227 KB opt-in shared memory per block

// Kernel parameters.  The kernel's rows are weight rows (M = N of the
// Linear), its columns the tokens (N = M of the Linear); Y is [tokens][M].
struct S8Params {
    const float* sx;        // [tokens] activation scales
    const float* sw;        // [M] weight scales
    const uint16_t* bias;   // bf16 [M] or null
    void* out;              // Y bf16 [tokens][M], or the int32 sums
    int M, N, K;
    int num_m;              // weight tiles of BM rows
    int k_stages;           // 128-K stages
    int k_split;            // units per tile, each over split_stages stages (1: no split)
    int split_stages;
    int num_tiles;          // work units: num_m * k_split
    int32_t* partial;       // k_split > 1: zeroed int32 sums [tokens][M]
    int32_t* counters;      // k_split > 1: zeroed arrivals, 4 per tile (one per 32-row group)
    int a_settled;          // the weights were complete before the previous kernel started
};

// ---------------------------------------------------------------------------
// Few-token post-scale GEMM on int8 operands.  The weights are the large
// operand of a few-token Linear and the whole cost at these sizes is their
// read, so this variant streams them as int8 (half the bytes of the 16-bit
// image).  One CTA per SM, no clusters: a CTA owns 128 weight rows (M = 128
// MMAs, cta_group::1), so a tile needs no other CTA and twice as many tiles
// feed the SMs.
// Roles (512 threads):
//   warp 0      producer: TMA of the slot's int8 weight tile and token image;
//   warp 1      TMEM allocation and the MMAs (kind::f16, fp16 operands);
//   warps 2-3   idle;
//   warps 4-11  converters, two warpgroups taking alternate stages.  A byte b
//               (two's complement x) becomes fp16 bits 0x6400 | (b ^ 0x80),
//               i.e. 1024 + x + 128, and subtracting 1152 leaves x exactly;
//               one byte permute builds two such halves and one packed fp16
//               subtraction finishes them;
//   warps 12-15 epilogue, one per TMEM lane quarter, all BN columns each
//               (chunk folds into int32, then Y or the split-K sums).
// A weight stage widened in shared memory for the MMA to read costs three
// shared-memory passes of its 16-bit form; written to tensor memory it costs
// none, and the tokens, widened once by s8_prep_kernel, arrive by TMA.
// ---------------------------------------------------------------- few tokens on int8 weight codes
//
// gemm_s8_kernel: Y[t][n] for at most 96 tokens, reading each int8 weight
// code once.  The kernel's rows are weight rows n (128 per tile, one CTA per
// tile and K split), its columns the tokens (BN >= tokens: one column tile).
// Each 128-K stage:
//   - TMA brings the int8 weight tile [128 rows x 128 bytes] and the fp16
//     image of the tokens [BN rows x 128 K] (two 64-element boxes), both with
//     the 128-byte swizzle, into one shared-memory slot;
//   - a converter warpgroup widens the weight tile into tensor memory, one
//     weight row per thread (64 columns of fp16 pairs, tcgen05.st);
//   - one thread issues eight tcgen05.mma with A in tensor memory and B in
//     shared memory; their commit frees the slot and the tensor-memory stage
//     of the same index (one ring: the producer's wait for a free slot also
//     orders the converters' next writes of that tensor-memory stage after
//     the MMAs that read it).
// fp16 holds every int8 value exactly, and within a chunk of eight stages
// (1024 K, |sum| <= 127 * 127 * 1024 < 2^24) the fp32 accumulation is exact;
// the epilogue folds each chunk into int32.  With K split, each unit adds its
// int32 sums into a zeroed buffer with integer atomics (exact in any order)
// and the warp whose arrival completes a 32-row group writes that group's Y.
// Two converter warpgroups take alternate stages, each with its own full
// barrier per slot (see the barrier layout in the kernel).  The producer asks
// each weight tile into L2 1024 K before its load.
constexpr int S8_BK = 128;                   // K per stage (bytes of an int8 weight row)
constexpr int S8_CHUNK_STAGES = 8;           // 1024 K per exact fp32 chunk
constexpr uint32_t S8_A_BYTES = BM * S8_BK;  // 16 KB
constexpr int S8_SPLIT_MAX_TILES = 76;       // K splits only when the weight rows make at most this many tiles
constexpr int S8_SPLIT_MAX = 8;
constexpr int S8_PREFETCH = 8;               // weight stages asked into L2 ahead of their load (1024 K)

template <int BN_>
struct CfgS8 {
    static constexpr int BN = BN_;
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 128, "token tile");
    static constexpr uint32_t B_BOX_BYTES = BN * 128;    // BN rows x 64 fp16
    static constexpr uint32_t B_BYTES = 2 * B_BOX_BYTES;
    static constexpr uint32_t SLOT = S8_A_BYTES + B_BYTES;
    static constexpr uint32_t A_TMEM0 = 2 * BN;          // after the two accumulator buffers
    static constexpr uint32_t SX_BYTES = 512;            // the tile's token scales
    static constexpr uint32_t BAR_BYTES = 512;
    static constexpr uint32_t RING_BUDGET = MAX_DYN_SMEM - 1024 - SX_BYTES - BAR_BYTES;
    // stages: shared-memory slots and 64-column tensor-memory stages alike
    static constexpr int S_SMEM = int(RING_BUDGET / SLOT);
    static constexpr int S_TMEM = int((TMEM_COLS - A_TMEM0) / 64);
    static constexpr int S = S_SMEM < S_TMEM ? S_SMEM : S_TMEM;
    static_assert(S >= 3 && A_TMEM0 + 64 * S <= TMEM_COLS, "ring");
    static_assert(4 * S + 5 <= int(BAR_BYTES / 8) - 1 && 2 * S <= 32, "barrier area, barrier bitmasks");
    static constexpr size_t SMEM = 1024 + size_t(S) * SLOT + SX_BYTES + BAR_BYTES;
    static constexpr uint32_t IDESC = idesc_f16_f32(BM, BN);
    static constexpr int LDW = 16;  // tensor-memory loads of 16 columns: the 128 int32 sums stay in registers
    static constexpr int GROUPS = BN / LDW;
};

// 16 int8 -> 16 fp16 (exact), as two 16-byte groups: the byte b ^ 0x80 goes
// under the exponent of 1024 (0x64xx is 1024 + (b ^ 0x80)) and 1152 comes off.
__device__ __forceinline__ void s8x16_to_f16(const uint4& v, uint4& lo, uint4& hi) {
    const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t p0 = __byte_perm(w[i], 0x64646464u, 0x4140);  // halves 1024 + u0, 1024 + u1
        const uint32_t p1 = __byte_perm(w[i], 0x64646464u, 0x4342);  // halves 1024 + u2, 1024 + u3
        __half2 h0 = __hsub2(*reinterpret_cast<const __half2*>(&p0), bias);
        __half2 h1 = __hsub2(*reinterpret_cast<const __half2*>(&p1), bias);
        o[2 * i] = *reinterpret_cast<uint32_t*>(&h0);
        o[2 * i + 1] = *reinterpret_cast<uint32_t*>(&h1);
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// Bring a 2-D tile of the tensor into L2 ahead of its load (no shared-memory
// destination, nothing to wait for): the weight stream of these kernels is
// latency-bound with a ring of a few stages, and loads that hit L2 keep it full.
__device__ __forceinline__ void tma_prefetch_l2_2d(const void* tmap, int32_t c0, int32_t c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(c0), "r"(c1)
                 : "memory");
}

// Widen weight row r of an int8 stage (128 rows x 128 bytes, as TMA wrote it
// with the 128-byte swizzle: 16-byte unit c of row r sits at unit c ^ (r & 7))
// into tensor memory at taddr (this warp's lane quarter, the stage's first
// column): 64 columns of fp16 pairs, element 2j in the low half of column j,
// the layout tcgen05.mma reads an A operand from tensor memory in.  The eight
// threads of a quarter-warp read eight different bank groups.
__device__ __forceinline__ void widen_row_to_tmem(const uint8_t* stage, int r, uint32_t taddr) {
    const uint8_t* row = stage + r * S8_BK;
    const int sw = r & 7;
    uint4 v[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) v[c] = *reinterpret_cast<const uint4*>(row + ((c ^ sw) << 4));
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t o[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint4 lo, hi;
            s8x16_to_f16(v[4 * h + c], lo, hi);
            o[8 * c + 0] = lo.x;
            o[8 * c + 1] = lo.y;
            o[8 * c + 2] = lo.z;
            o[8 * c + 3] = lo.w;
            o[8 * c + 4] = hi.x;
            o[8 * c + 5] = hi.y;
            o[8 * c + 6] = hi.z;
            o[8 * c + 7] = hi.w;
        }
        tmem_st_32x32b_x32(taddr + 32 * h, o);
    }
}

// Output column n (a weight row) for the BN tokens of the tile:
// y = ((float(acc) * sx[t]) * sw[n]) + bias[n], the operation order of every
// other post-scale epilogue, or the int32 sums themselves.  Lanes hold
// consecutive n, so each token's stores are contiguous.
template <int EPI, int BN>
__device__ __forceinline__ void s8_store(const int32_t (&acc)[BN], const S8Params& p, int n, const float* sxs,
                                         float swn, float bn) {
    if (n >= p.M) return;
    if constexpr (EPI == kEpiPostscaleS32) {
        int32_t* out = static_cast<int32_t*>(p.out) + n;
#pragma unroll
        for (int t = 0; t < BN; ++t) {
            if (t < p.N) *out = acc[t];
            out += p.M;
        }
    } else {
        // 16 tokens at a time: the scales are read before any of the group's
        // stores (the compiler cannot tell shared and global memory apart here)
        uint16_t* out = static_cast<uint16_t*>(p.out) + n;
#pragma unroll
        for (int g = 0; g < BN; g += 16) {
            if (g >= p.N) break;
            float sv[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) sv[e] = sxs[g + e];
            uint32_t y[8];  // two tokens' bf16 per register: one paired conversion
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
                float v0 = __fmul_rn(__fmul_rn(__int2float_rn(acc[g + e]), sv[e]), swn);
                float v1 = __fmul_rn(__fmul_rn(__int2float_rn(acc[g + e + 1]), sv[e + 1]), swn);
                if (p.bias) {
                    v0 = __fadd_rn(v0, bn);
                    v1 = __fadd_rn(v1, bn);
                }
                __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
                y[e / 2] = *reinterpret_cast<uint32_t*>(&h);
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                if (g + e < p.N) *out = static_cast<uint16_t>(y[e / 2] >> (16 * (e & 1)));
                out += p.M;
            }
        }
    }
}

enum WaitSiteS8 : int {
    kSiteS8ProducerEmpty = 11,
    kSiteS8ConvFull = 12,
    kSiteS8MmaFull = 14,
    kSiteS8ProducerDrain = 15,
    kSiteS8MmaAccEmpty = 16,
    kSiteS8EpiAccFull = 17,
    kSiteS8MmaDrain = 18,
};

constexpr int S8_CONV_GROUPS = 2;                        // converter warpgroups
constexpr int S8_EPI_WARP0 = 4 + 4 * S8_CONV_GROUPS;     // first epilogue warp
constexpr int S8_THREADS = 32 * (S8_EPI_WARP0 + 4);
// Register split: warpgroup 0 (producer, MMA) 56, converters 80, epilogue 232,
// within the launch budget of S8_THREADS x 128 (512 threads at 128).
static_assert(128 * 56 + 128 * S8_CONV_GROUPS * 80 + 128 * 232 <= S8_THREADS * (65536 / S8_THREADS),
              "int8 kernel register split exceeds the launch budget");

// Work unit u of the int8 kernel: weight tile mb, K stages [ks0, ks1).
__device__ __forceinline__ void s8_unit(int u, const S8Params& p, int& mb, int& ks0, int& ks1) {
    mb = u / p.k_split;
    ks0 = (u - mb * p.k_split) * p.split_stages;
    ks1 = min(p.k_stages, ks0 + p.split_stages);
}

template <int EPI, int BN>
__global__ void __launch_bounds__(S8_THREADS, 1)
    gemm_s8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const S8Params p) {
    grid_launch_dependents();
    using C = CfgS8<BN>;
    constexpr int S = C::S;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* sxs = reinterpret_cast<float*>(ring + S * C::SLOT);
    // full8[g * S + s]: the copies of slot s for a stage of converter group g.
    // The groups take alternate stages and S may be odd, so a slot serves
    // both groups in turn; with one barrier per slot a group would wait on
    // only every other phase of it, and a parity wait cannot tell the other
    // group's earlier phase still in flight (copies land out of order) from
    // its own phase complete.  One barrier per slot and group lets every
    // waiter see every phase of the barriers it waits on.
    uint64_t* full8 = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sxs) + C::SX_BYTES);
    uint64_t* full16 = full8 + 2 * S;
    uint64_t* empty = full16 + S;
    uint64_t* acc_full = empty + S;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* mma_drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = static_cast<int>(blockIdx.x);
    const int nctas = static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full8[s], 1);       // the producer's arrive + the slot's bytes (group 0)
            mbar_init(&full8[S + s], 1);   // (group 1)
            mbar_init(&full16[s], 4);      // the four converter warps of the stage's group
            mbar_init(&empty[s], 1);       // the MMA commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);  // the four epilogue warps
        }
        mbar_init(mma_drain, 1);
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Weights settled before the previous kernel started may be read before
    // the dependency wait (the producer's first fills); nothing else is.
    if (warp != 0) grid_dependency_wait();
    const uint32_t tmem_base = *tmem_slot;
    if (warp < 4) {
      regs_dec<56>();
      if (warp == 0) {
        // ------------------------------------------------------------ producer
        const bool elected = elect_one_sync();
        int pre = 0;
        if (elected && p.a_settled && cta < p.num_tiles) {
            int mb, ks0, ks1;
            s8_unit(cta, p, mb, ks0, ks1);
            pre = min(S, ks1 - ks0);
            for (int i = 0; i < pre; ++i) {
                uint64_t* bar = &full8[(i % S8_CONV_GROUPS) * S + i];
                mbar_arrive_expect_tx(bar, C::SLOT);
                tma_load_2d(ring + i * C::SLOT, &tmA, bar, (ks0 + i) * S8_BK, mb * BM);
            }
            for (int i = pre; i < min(S8_PREFETCH, ks1 - ks0); ++i)
                tma_prefetch_l2_2d(&tmA, (ks0 + i) * S8_BK, mb * BM);
        }
        grid_dependency_wait();
        if (elected) {
            int stage = 0;
            uint32_t phase = 0;
            int g_stage = 0;                        // stage count of this CTA (all its units)
            uint32_t uses = 0;                      // bit b: parity of the uses of full8[b] so far
            uint32_t armed = 0, armed_phase = 0;    // per full8 barrier: used, and its last use's parity
            bool ok = true;
            for (int u = cta; ok && u < p.num_tiles; u += nctas) {
                int mb, ks0, ks1;
                s8_unit(u, p, mb, ks0, ks1);
                if (!(u == cta && pre > 0))
                    for (int i = S; i < min(S8_PREFETCH, ks1 - ks0); ++i)
                        tma_prefetch_l2_2d(&tmA, (ks0 + i) * S8_BK, mb * BM);
                for (int ks = ks0; ks < ks1; ++ks, ++g_stage) {
                    uint8_t* slot = ring + stage * C::SLOT;
                    const int b = (g_stage % S8_CONV_GROUPS) * S + stage;
                    if (ks + S8_PREFETCH < ks1) tma_prefetch_l2_2d(&tmA, (ks + S8_PREFETCH) * S8_BK, mb * BM);
                    if (!(u == cta && ks - ks0 < pre)) {
                        if (!mbar_wait(&empty[stage], phase ^ 1u, kSiteS8ProducerEmpty)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&full8[b], C::SLOT);
                        tma_load_2d(slot, &tmA, &full8[b], ks * S8_BK, mb * BM);
                    }
                    tma_load_2d(slot + S8_A_BYTES, &tmB, &full8[b], ks * S8_BK, 0);
                    tma_load_2d(slot + S8_A_BYTES + C::B_BOX_BYTES, &tmB, &full8[b], ks * S8_BK + 64, 0);
                    armed |= 1u << b;
                    armed_phase = (armed_phase & ~(1u << b)) | (((uses >> b) & 1u) << b);
                    uses ^= 1u << b;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Every copy issued has landed before this CTA's shared memory is released.
            for (int b = 0; b < S8_CONV_GROUPS * S; ++b)
                if (armed & (1u << b)) mbar_wait(&full8[b], (armed_phase >> b) & 1u, kSiteS8ProducerDrain);
        }
      } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (elect_one_sync()) {
            int stage = 0;
            uint32_t phase = 0;
            int buf = 0;
            uint32_t buf_phase = 0;
            bool ok = true;
            // B descriptor of slot 0 (start address in bits 0-13, in 16-byte units)
            const uint64_t desc0 = smem_desc_kmajor_sw128(smem_u32(ring + S8_A_BYTES));
            for (int u = cta; ok && u < p.num_tiles; u += nctas) {
                int mb, ks0, ks1;
                s8_unit(u, p, mb, ks0, ks1);
                const int nchunks = (ks1 - ks0 + S8_CHUNK_STAGES - 1) / S8_CHUNK_STAGES;
                for (int c = 0; ok && c < nchunks; ++c) {
                    if (!mbar_wait(&acc_empty[buf], buf_phase ^ 1u, kSiteS8MmaAccEmpty)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
                    const int s0 = ks0 + c * S8_CHUNK_STAGES;
                    const int s1 = min(ks1, s0 + S8_CHUNK_STAGES);
                    for (int ks = s0; ks < s1; ++ks) {
                        // the widened weights; the converters waited for the slot's copies
                        // (the token image the MMA reads from it) before arriving
                        if (!mbar_wait(&full16[stage], phase, kSiteS8MmaFull)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_tmem = tmem_base + C::A_TMEM0 + static_cast<uint32_t>(stage * 64);
                        const uint64_t db = desc0 + static_cast<uint64_t>((stage * C::SLOT) >> 4);
                        mma_f16_ts(d_tmem, a_tmem, db, C::IDESC, ks > s0 ? 1u : 0u);
#pragma unroll
                        for (int k = 1; k < S8_BK / 16; ++k)
                            mma_f16_ts(d_tmem, a_tmem + k * 8,
                                       db + static_cast<uint64_t>(((k >> 2) * C::B_BOX_BYTES + (k & 3) * 32) >> 4),
                                       C::IDESC, 1u);
                        mma_commit(&empty[stage]);
                        if (++stage == S) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    mma_commit(&acc_full[buf]);
                    buf ^= 1;
                    if (buf == 0) buf_phase ^= 1u;
                }
            }
            mma_commit(mma_drain);
            mbar_wait(mma_drain, 0, kSiteS8MmaDrain);
        }
      }
    } else if (warp < S8_EPI_WARP0) {
        regs_dec<80>();
        // ------------------------------------------------------------ converters (warps 4..S8_EPI_WARP0-1)
        const int group = (warp - 4) >> 2;     // converter warpgroup
        const int r = ((warp & 3) << 5) | lane;  // weight row of the tile = tensor-memory lane
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16) + C::A_TMEM0;
        int stage = 0;
        int g_stage = 0;                       // stage count of this CTA (all its units)
        uint32_t uses = 0;                     // bit s: parity of this group's uses of full8[group * S + s]
        bool ok = true;
        for (int u = cta; ok && u < p.num_tiles; u += nctas) {
            int mb, ks0, ks1;
            s8_unit(u, p, mb, ks0, ks1);
            for (int ks = ks0; ks < ks1; ++ks, ++g_stage) {
                if (g_stage % S8_CONV_GROUPS == group) {
                    // the slot's copies landed, so the MMAs that last read this
                    // tensor-memory stage have completed (their commit freed the slot)
                    if (!mbar_wait(&full8[group * S + stage], (uses >> stage) & 1u, kSiteS8ConvFull)) {
                        ok = false;
                        break;
                    }
                    uses ^= 1u << stage;
                    tc_fence_after();
                    widen_row_to_tmem(ring + stage * C::SLOT, r, lane_base + static_cast<uint32_t>(stage * 64));
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&full16[stage]);
                }
                if (++stage == S) stage = 0;
            }
        }
    } else {
        regs_inc<232>();
        // ------------------------------------------------------------ epilogue (the last four warps)
        constexpr int LDW = C::LDW;
        constexpr int GROUPS = C::GROUPS;
        const int quarter = warp & 3;
        const int et = static_cast<int>(threadIdx.x) - 32 * S8_EPI_WARP0;  // 0..127
        if (et < BN) sxs[et] = (EPI == kEpiPostscaleBf16 && et < p.N) ? __ldg(p.sx + et) : 0.0f;
        named_bar_sync(1, 128);  // the four epilogue warps
        int buf = 0;
        uint32_t buf_phase = 0;
        bool ok = true;
        for (int u = cta; ok && u < p.num_tiles; u += nctas) {
            int mb, ks0, ks1;
            s8_unit(u, p, mb, ks0, ks1);
            const int nchunks = (ks1 - ks0 + S8_CHUNK_STAGES - 1) / S8_CHUNK_STAGES;
            const int n = mb * BM + quarter * 32 + lane;  // output column (weight row)
            float swn = 0.0f, bn = 0.0f;
            if (EPI == kEpiPostscaleBf16 && n < p.M) {
                swn = __ldg(p.sw + n);
                if (p.bias) bn = __uint_as_float(static_cast<uint32_t>(__ldg(p.bias + n)) << 16);
            }
            int32_t acc[BN];
#pragma unroll
            for (int e = 0; e < BN; ++e) acc[e] = 0;
            for (int c = 0; c < nchunks; ++c) {
                if (!mbar_wait(&acc_full[buf], buf_phase, kSiteS8EpiAccFull)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr =
                    tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(buf * BN);
                uint32_t ra[LDW], rb[LDW];
                tmem_ld_32x32b_x16(taddr, ra);
                tmem_wait_ld_regs(ra);
#pragma unroll
                for (int j = 0; j < GROUPS; ++j) {
                    uint32_t(&cur)[LDW] = (j & 1) ? rb : ra;
                    uint32_t(&nxt)[LDW] = (j & 1) ? ra : rb;
                    if (j + 1 < GROUPS) tmem_ld_32x32b_x16(taddr + (j + 1) * LDW, nxt);
#pragma unroll
                    for (int e = 0; e < LDW; ++e) acc[j * LDW + e] += __float2int_rz(__uint_as_float(cur[e]));
                    if (j + 1 < GROUPS) tmem_wait_ld_regs(nxt);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[buf]);
                buf ^= 1;
                if (buf == 0) buf_phase ^= 1u;
            }
            if (!ok) break;
            if (p.k_split == 1) {
                s8_store<EPI, BN>(acc, p, n, sxs, swn, bn);
            } else {
                // add this unit's sums; the warp completing the row group writes it
                if (n < p.M) {
                    int32_t* dst = p.partial + n;  // [token][weight row]: stepped by one row of sums
#pragma unroll
                    for (int t = 0; t < BN; ++t) {
                        if (t < p.N) atomicAdd(dst, acc[t]);
                        dst += p.M;
                    }
                }
                __threadfence();
                __syncwarp();
                int arrived = 0;
                if (lane == 0) arrived = atomicAdd(p.counters + mb * 4 + quarter, 1);
                arrived = __shfl_sync(0xffffffffu, arrived, 0);
                if (arrived == p.k_split - 1) {
                    __threadfence();
                    if (n < p.M) {
                        const int32_t* src = p.partial + n;
#pragma unroll
                        for (int t = 0; t < BN; ++t) {
                            if (t < p.N) acc[t] = __ldcg(src);
                            src += p.M;
                        }
                    }
                    s8_store<EPI, BN>(acc, p, n, sxs, swn, bn);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// First step of the int8-operand GEMM: the fp16 image of the tokens' codes
// (the MMA's B operand) and, when K is split, zeroed int32 sums and arrival
// counters.  It lets the GEMM launch at once (the GEMM's prologue and its
// first weight loads overlap this kernel) and waits for its own predecessor,
// which may be writing Xq.
__global__ void __launch_bounds__(256) s8_prep_kernel(const uint4* __restrict__ xq, int64_t n16,
                                                      uint4* __restrict__ img, uint4* __restrict__ zero,
                                                      int64_t nz16) {
    grid_launch_dependents();
    grid_dependency_wait();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (int64_t i = i0; i < n16; i += stride) {
        uint4 lo, hi;
        s8x16_to_f16(__ldg(xq + i), lo, hi);
        img[2 * i] = lo;
        img[2 * i + 1] = hi;
    }
    for (int64_t i = i0; i < nz16; i += stride) zero[i] = make_uint4(0u, 0u, 0u, 0u);
}

// ---------------------------------------------------------------- 97..288 tokens on int8 weight codes
//
// gemm_s8w_kernel: the same product for 97..288 tokens.  Two accumulators of
// the whole token tile no longer fit in tensor memory beside the widened
// weights, and one alone would stop the MMAs at every 1024-K chunk while the
// epilogue folds it into int32.  So the tile is cut into P token parts of W
// columns (P = 3 at 288 tokens, else 2; one MMA of N = W per part) that
// share P + 1 accumulator regions of W columns: the parts' chunks end at
// staggered stages (s8w_chunk_start), and at the end of a chunk a part moves
// on into the free region while the epilogue folds the one it leaves.  The
// MMAs never wait for a fold as long as it ends within the 16 / P stages
// before the next part's chunk ends.  (Smaller parts cost more than they
// save: a tcgen05.mma of N <= ~112 takes about as long as one of N = 112.)  The token image of a 128-K stage would take 72 KB at
// BN = 288, so stages are 64 K wide: the int8 weight tile [128 rows x 64
// bytes] arrives with the 64-byte swizzle and the token image [BN rows x 64
// K] as P boxes of W rows with the 128-byte swizzle.
// Roles (512 threads):
//   warp 0      producer;  warp 1  TMEM allocation and the MMAs;  warps 2-3 idle;
//   warps 4-7   converters, one weight row per thread (32 columns of fp16 pairs);
//   warps 8-15  epilogue: warp 8 + 4c + q holds tensor-memory lane quarter q
//               and column half c of every part (BN / 2 int32 sums per thread),
//               and all eight fold each region the MMAs leave.
constexpr int S8W_BK = 64;                      // K per stage (bytes of an int8 weight row)
constexpr int S8W_CHUNK_STAGES = 16;            // 1024 K per exact fp32 chunk
constexpr int S8W_PREFETCH = 16;                // weight stages asked into L2 ahead of their load (1024 K)
constexpr uint32_t S8W_A_BYTES = BM * S8W_BK;   // 8 KB
constexpr int S8W_THREADS = 512;
constexpr int S8W_EPI_WARP0 = 8;
// Register split: warpgroup 0 64 (the MMA issuer's region bookkeeping), converters 64, the two
// epilogue warpgroups 192 (up to 144 int32 sums per thread).
static_assert(128 * 64 + 128 * 64 + 256 * 192 <= 65536, "wide int8 kernel register split exceeds the launch budget");

// Token parts of a wide token tile of bn columns.
__host__ __device__ constexpr int s8w_parts(int bn) { return bn > 256 ? 3 : 2; }

template <int BN_>
struct CfgS8W {
    static constexpr int BN = BN_;
    static constexpr int P = s8w_parts(BN);             // token parts
    static constexpr int W = BN / P;                    // tokens per part: N of its MMA, columns of a region
    static constexpr int REGIONS = P + 1;
    static constexpr int HALF = W / 2;                  // columns of a region per epilogue warp
    static_assert(BN % (16 * P) == 0 && W >= 64 && W <= 128 && HALF % 8 == 0 && P <= 4, "wide token tile");
    static constexpr uint32_t B_PART_BYTES = W * 128;   // W rows x 64 fp16, a multiple of the 1024-byte swizzle atom
    static constexpr uint32_t SLOT = S8W_A_BYTES + P * B_PART_BYTES;
    static constexpr uint32_t A_TMEM0 = REGIONS * W;    // after the accumulator regions
    static constexpr uint32_t SX_BYTES = 2048;          // the tile's token scales
    static constexpr uint32_t BAR_BYTES = 512;
    static constexpr uint32_t RING_BUDGET = MAX_DYN_SMEM - 1024 - SX_BYTES - BAR_BYTES;
    static constexpr int S_SMEM = int(RING_BUDGET / SLOT);
    static constexpr int S_TMEM = int((TMEM_COLS - A_TMEM0) / 32);
    static constexpr int S = S_SMEM < S_TMEM ? S_SMEM : S_TMEM;
    static_assert(S >= 4 && A_TMEM0 + 32 * S <= TMEM_COLS, "ring");
    static_assert(3 * S + 2 * REGIONS + 1 <= int(BAR_BYTES / 8) - 1, "barrier area");
    static_assert(BN * 4 <= int(SX_BYTES), "scale area");
    static constexpr size_t SMEM = 1024 + size_t(S) * SLOT + SX_BYTES + BAR_BYTES;
    static constexpr uint32_t IDESC = idesc_f16_f32(BM, W);
};

// 32 lanes x 8 consecutive 32-bit columns, and the matching wait.
__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_ld_regs8(uint32_t (&r)[8]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7])
                 :
                 : "memory");
}

// Widen weight row r of a 64-K int8 stage (128 rows x 64 bytes, as TMA wrote
// it with the 64-byte swizzle: 16-byte unit c of row r sits at unit
// c ^ ((r >> 1) & 3)) into tensor memory at taddr: 32 columns of fp16 pairs.
// The eight threads of a quarter-warp read eight different bank groups.
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void widen_row64_to_tmem(const uint8_t* stage, int r, uint32_t taddr) {
    const uint8_t* row = stage + r * S8W_BK;
    const int sw = (r >> 1) & 3;
    uint4 v[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) v[c] = *reinterpret_cast<const uint4*>(row + ((c ^ sw) << 4));
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t o[16];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            uint4 lo, hi;
            s8x16_to_f16(v[2 * h + c], lo, hi);
            o[8 * c + 0] = lo.x;
            o[8 * c + 1] = lo.y;
            o[8 * c + 2] = lo.z;
            o[8 * c + 3] = lo.w;
            o[8 * c + 4] = hi.x;
            o[8 * c + 5] = hi.y;
            o[8 * c + 6] = hi.z;
            o[8 * c + 7] = hi.w;
        }
        tmem_st_32x32b_x16(taddr + 16 * h, o);
    }
}

// Output column n for the tokens t0 .. t0 + CNT - 1 (a part's columns held
// by one epilogue warp): the post-scale epilogue of s8_store, 8 tokens at a
// time, or the int32 sums.
template <int EPI, int CNT>
__device__ __forceinline__ void s8w_store(const int32_t (&acc)[CNT], const S8Params& p, int n, int t0,
                                          const float* sxs, float swn, float bn) {
    static_assert(CNT % 8 == 0, "token groups");
    if (n >= p.M) return;
    if constexpr (EPI == kEpiPostscaleS32) {
        int32_t* out = static_cast<int32_t*>(p.out) + static_cast<int64_t>(t0) * p.M + n;
#pragma unroll
        for (int t = 0; t < CNT; ++t) {
            if (t0 + t < p.N) *out = acc[t];
            out += p.M;
        }
    } else {
        uint16_t* out = static_cast<uint16_t*>(p.out) + static_cast<int64_t>(t0) * p.M + n;
#pragma unroll
        for (int g = 0; g < CNT; g += 8) {
            if (t0 + g >= p.N) break;
            float sv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) sv[e] = sxs[t0 + g + e];
            uint32_t y[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                float v0 = __fmul_rn(__fmul_rn(__int2float_rn(acc[g + e]), sv[e]), swn);
                float v1 = __fmul_rn(__fmul_rn(__int2float_rn(acc[g + e + 1]), sv[e + 1]), swn);
                if (p.bias) {
                    v0 = __fadd_rn(v0, bn);
                    v1 = __fadd_rn(v1, bn);
                }
                __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
                y[e / 2] = *reinterpret_cast<uint32_t*>(&h);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (t0 + g + e < p.N) *out = static_cast<uint16_t>(y[e / 2] >> (16 * (e & 1)));
                out += p.M;
            }
        }
    }
}

// Local stages of a work unit (of n) at which token part q of P starts an
// exact 1024-K chunk: stage 0, and every stage j with (j + q * (16 / P)) a
// multiple of 16 -- so part 0 at 16, 32, ...; with two parts part 1 at 8,
// 24, ...; with three parts part 1 at 11, 27, ... and part 2 at 6, 22, ...
// No two parts start a chunk at the same stage after stage 0.
template <int P>
__device__ __forceinline__ bool s8w_chunk_start(int q, int j) {
    return j == 0 || (j + q * (S8W_CHUNK_STAGES / P)) % S8W_CHUNK_STAGES == 0;
}
// The part whose chunk starts at local stage j > 0, or -1.
template <int P>
__device__ __forceinline__ int s8w_part_starting(int j) {
#pragma unroll
    for (int q = 0; q < P; ++q)
        if ((j + q * (S8W_CHUNK_STAGES / P)) % S8W_CHUNK_STAGES == 0) return q;
    return -1;
}

enum WaitSiteS8W : int {
    kSiteS8WProducerEmpty = 21,
    kSiteS8WConvFull = 22,
    kSiteS8WMmaFull = 23,
    kSiteS8WProducerDrain = 24,
    kSiteS8WMmaAccEmpty = 25,
    kSiteS8WEpiAccFull = 26,
    kSiteS8WMmaDrain = 27,
};

// Fold a region's chunk into one warp's int32 sums: HALF columns from taddr,
// 8 at a time, the next load in flight while the last is converted.
template <int HALF>
__device__ __forceinline__ void s8w_fold(int32_t (&acc)[HALF], uint32_t taddr) {
    constexpr int G = HALF / 8;
    uint32_t ra[8], rb[8];
    tmem_ld_32x32b_x8(taddr, ra);
    tmem_wait_ld_regs8(ra);
#pragma unroll
    for (int j = 0; j < G; ++j) {
        uint32_t(&cur)[8] = (j & 1) ? rb : ra;
        uint32_t(&nxt)[8] = (j & 1) ? ra : rb;
        if (j + 1 < G) tmem_ld_32x32b_x8(taddr + (j + 1) * 8, nxt);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[j * 8 + e] += __float2int_rz(__uint_as_float(cur[e]));
        if (j + 1 < G) tmem_wait_ld_regs8(nxt);
    }
}

// Region of token part q in a packed table (four bits per part), and the
// table after part q moves into region r.
__device__ __forceinline__ int s8w_region(uint32_t table, int q) { return static_cast<int>((table >> (4 * q)) & 15u); }
__device__ __forceinline__ uint32_t s8w_move(uint32_t table, int q, int r) {
    return (table & ~(15u << (4 * q))) | (static_cast<uint32_t>(r) << (4 * q));
}
// The starting table: part q in region q (region P is free).
template <int P>
__host__ __device__ constexpr uint32_t s8w_table0() {
    uint32_t t = 0;
    for (int q = 0; q < P; ++q) t |= static_cast<uint32_t>(q) << (4 * q);
    return t;
}

template <int EPI, int BN>
__global__ void __launch_bounds__(S8W_THREADS, 1)
    gemm_s8w_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const S8Params p) {
    grid_launch_dependents();
    using C = CfgS8W<BN>;
    constexpr int S = C::S;
    constexpr int P = C::P;
    constexpr int W = C::W;
    constexpr int HALF = C::HALF;
    constexpr uint32_t TABLE0 = s8w_table0<P>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* sxs = reinterpret_cast<float*>(ring + S * C::SLOT);
    uint64_t* full8 = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sxs) + C::SX_BYTES);
    uint64_t* full16 = full8 + S;
    uint64_t* empty = full16 + S;
    uint64_t* acc_full = empty + S;  // per accumulator region
    uint64_t* acc_empty = acc_full + C::REGIONS;
    uint64_t* mma_drain = acc_empty + C::REGIONS;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = static_cast<int>(blockIdx.x);
    const int nctas = static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full8[s], 1);   // the producer's arrive + the slot's bytes
            mbar_init(&full16[s], 4);  // the four converter warps
            mbar_init(&empty[s], 1);   // the MMA commit
        }
        for (int r = 0; r < C::REGIONS; ++r) {
            mbar_init(&acc_full[r], 1);   // the MMA commit at the end of a part's chunk
            mbar_init(&acc_empty[r], 8);  // the eight epilogue warps, after the fold
        }
        mbar_init(mma_drain, 1);
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp != 0) grid_dependency_wait();
    const uint32_t tmem_base = *tmem_slot;
    if (warp < 4) {
      regs_dec<64>();
      if (warp == 0) {
        // ------------------------------------------------------------ producer
        const bool elected = elect_one_sync();
        int pre = 0;
        if (elected && p.a_settled && cta < p.num_tiles) {
            int mb, ks0, ks1;
            s8_unit(cta, p, mb, ks0, ks1);
            pre = min(S, ks1 - ks0);
            for (int i = 0; i < pre; ++i) {
                mbar_arrive_expect_tx(&full8[i], C::SLOT);
                tma_load_2d(ring + i * C::SLOT, &tmA, &full8[i], (ks0 + i) * S8W_BK, mb * BM);
            }
            for (int i = pre; i < min(S8W_PREFETCH, ks1 - ks0); ++i)
                tma_prefetch_l2_2d(&tmA, (ks0 + i) * S8W_BK, mb * BM);
        }
        grid_dependency_wait();
        if (elected) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_phase = 0;
            bool ok = true;
            for (int u = cta; ok && u < p.num_tiles; u += nctas) {
                int mb, ks0, ks1;
                s8_unit(u, p, mb, ks0, ks1);
                if (!(u == cta && pre > 0))
                    for (int i = S; i < min(S8W_PREFETCH, ks1 - ks0); ++i)
                        tma_prefetch_l2_2d(&tmA, (ks0 + i) * S8W_BK, mb * BM);
                for (int ks = ks0; ks < ks1; ++ks) {
                    uint8_t* slot = ring + stage * C::SLOT;
                    if (ks + S8W_PREFETCH < ks1) tma_prefetch_l2_2d(&tmA, (ks + S8W_PREFETCH) * S8W_BK, mb * BM);
                    if (!(u == cta && ks - ks0 < pre)) {
                        if (!mbar_wait(&empty[stage], phase ^ 1u, kSiteS8WProducerEmpty)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&full8[stage], C::SLOT);
                        tma_load_2d(slot, &tmA, &full8[stage], ks * S8W_BK, mb * BM);
                    }
#pragma unroll
                    for (int q = 0; q < P; ++q)
                        tma_load_2d(slot + S8W_A_BYTES + q * C::B_PART_BYTES, &tmB, &full8[stage], ks * S8W_BK,
                                    q * W);
                    armed |= 1u << stage;
                    armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int s = 0; s < S; ++s)
                if (armed & (1u << s)) mbar_wait(&full8[s], (armed_phase >> s) & 1u, kSiteS8WProducerDrain);
        }
      } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (elect_one_sync()) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t table = TABLE0;  // region of each part
            int free_r = P;           // the region no part uses
            uint32_t used = 0;        // bit r: parity of the chunks committed to region r
            bool ok = true;
            const uint64_t desc0 = smem_desc_kmajor_sw128(smem_u32(ring + S8W_A_BYTES));
            for (int u = cta; ok && u < p.num_tiles; u += nctas) {
                int mb, ks0, ks1;
                s8_unit(u, p, mb, ks0, ks1);
                const int n = ks1 - ks0;
                // every region a part starts in has been folded (the previous unit's last chunks)
#pragma unroll
                for (int q = 0; q < P; ++q) {
                    const int r = s8w_region(table, q);
                    ok = ok && mbar_wait(&acc_empty[r], ((used >> r) & 1u) ^ 1u, kSiteS8WMmaAccEmpty);
                }
                if (!ok) break;
                tc_fence_after();
                for (int j = 0; j < n; ++j) {
                    const int qs = j > 0 ? s8w_part_starting<P>(j) : -1;
                    if (qs >= 0) {
                        // part qs's chunk is complete: the epilogue folds its region while
                        // the part goes on in the free one, once that one's last fold is done
                        const int old = s8w_region(table, qs);
                        mma_commit(&acc_full[old]);
                        used ^= 1u << old;
                        table = s8w_move(table, qs, free_r);
                        const int r = free_r;
                        free_r = old;
                        if (!mbar_wait(&acc_empty[r], ((used >> r) & 1u) ^ 1u, kSiteS8WMmaAccEmpty)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    if (!mbar_wait(&full16[stage], phase, kSiteS8WMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_tmem = tmem_base + C::A_TMEM0 + static_cast<uint32_t>(stage * 32);
                    const uint64_t db = desc0 + static_cast<uint64_t>((stage * C::SLOT) >> 4);
#pragma unroll
                    for (int q = 0; q < P; ++q) {
                        const uint32_t d = tmem_base + static_cast<uint32_t>(s8w_region(table, q) * W);
                        const uint32_t first = s8w_chunk_start<P>(q, j) ? 0u : 1u;
#pragma unroll
                        for (int k = 0; k < S8W_BK / 16; ++k)
                            mma_f16_ts(d, a_tmem + k * 8,
                                       db + static_cast<uint64_t>((q * C::B_PART_BYTES + k * 32) >> 4), C::IDESC,
                                       k > 0 ? 1u : first);
                    }
                    mma_commit(&empty[stage]);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                // the parts' last chunks of the unit
#pragma unroll
                for (int q = 0; q < P; ++q) {
                    const int r = s8w_region(table, q);
                    mma_commit(&acc_full[r]);
                    used ^= 1u << r;
                }
            }
            mma_commit(mma_drain);
            mbar_wait(mma_drain, 0, kSiteS8WMmaDrain);
        }
      }
    } else if (warp < S8W_EPI_WARP0) {
        regs_dec<64>();
        // ------------------------------------------------------------ converters (warps 4..7)
        const int r = ((warp & 3) << 5) | lane;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16) + C::A_TMEM0;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int u = cta; ok && u < p.num_tiles; u += nctas) {
            int mb, ks0, ks1;
            s8_unit(u, p, mb, ks0, ks1);
            for (int ks = ks0; ks < ks1; ++ks) {
                // the slot's copies landed, so the MMAs that last read this
                // tensor-memory stage have completed (their commit freed the slot)
                if (!mbar_wait(&full8[stage], phase, kSiteS8WConvFull)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                widen_row64_to_tmem(ring + stage * C::SLOT, r, lane_base + static_cast<uint32_t>(stage * 32));
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&full16[stage]);
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else {
        regs_inc<192>();
        // ------------------------------------------------------------ epilogue (warps 8..15)
        const int quarter = warp & 3;
        const int ch = (warp - S8W_EPI_WARP0) >> 2;                       // column half of every part
        const int et = static_cast<int>(threadIdx.x) - 32 * S8W_EPI_WARP0;  // 0..255
        for (int i = et; i < BN; i += 256)
            sxs[i] = (EPI == kEpiPostscaleBf16 && i < p.N) ? __ldg(p.sx + i) : 0.0f;
        named_bar_sync(1, 256);  // the eight epilogue warps
        uint32_t table = TABLE0;  // the MMA issuer's region table, replayed
        int free_r = P;
        uint32_t folded = 0;      // bit r: parity of the folds of region r
        bool ok = true;
        const uint32_t lane_base =
            tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(ch * HALF);
        for (int u = cta; ok && u < p.num_tiles; u += nctas) {
            int mb, ks0, ks1;
            s8_unit(u, p, mb, ks0, ks1);
            const int n_st = ks1 - ks0;
            const int n = mb * BM + quarter * 32 + lane;  // output column (weight row)
            float swn = 0.0f, bn = 0.0f;
            if (EPI == kEpiPostscaleBf16 && n < p.M) {
                swn = __ldg(p.sw + n);
                if (p.bias) bn = __uint_as_float(static_cast<uint32_t>(__ldg(p.bias + n)) << 16);
            }
            int32_t acc[P][HALF];
#pragma unroll
            for (int q = 0; q < P; ++q)
#pragma unroll
                for (int e = 0; e < HALF; ++e) acc[q][e] = 0;
            // fold part q's chunk from region r into the part's sums
            auto fold = [&](int q, int r) -> bool {
                if (!mbar_wait(&acc_full[r], (folded >> r) & 1u, kSiteS8WEpiAccFull)) return false;
                folded ^= 1u << r;
                tc_fence_after();
                const uint32_t taddr = lane_base + static_cast<uint32_t>(r * W);
#pragma unroll
                for (int qq = 0; qq < P; ++qq)
                    if (qq == q) s8w_fold<HALF>(acc[qq], taddr);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[r]);
                return true;
            };
            for (int j = 1; ok && j < n_st; ++j) {
                const int qs = s8w_part_starting<P>(j);
                if (qs < 0) continue;
                const int old = s8w_region(table, qs);
                ok = fold(qs, old);
                table = s8w_move(table, qs, free_r);
                free_r = old;
            }
#pragma unroll
            for (int q = 0; q < P; ++q) ok = ok && fold(q, s8w_region(table, q));
            if (!ok) break;
            if (p.k_split == 1) {
#pragma unroll
                for (int q = 0; q < P; ++q) s8w_store<EPI, HALF>(acc[q], p, n, q * W + ch * HALF, sxs, swn, bn);
            } else {
                // add this unit's sums; the warp completing the (row group, column half) writes it
                if (n < p.M) {
#pragma unroll
                    for (int q = 0; q < P; ++q) {
                        const int t0 = q * W + ch * HALF;
                        int32_t* dst = p.partial + static_cast<int64_t>(t0) * p.M + n;
#pragma unroll
                        for (int t = 0; t < HALF; ++t) {
                            if (t0 + t < p.N) atomicAdd(dst, acc[q][t]);
                            dst += p.M;
                        }
                    }
                }
                __threadfence();
                __syncwarp();
                int arrived = 0;
                if (lane == 0) arrived = atomicAdd(p.counters + mb * 8 + ch * 4 + quarter, 1);
                arrived = __shfl_sync(0xffffffffu, arrived, 0);
                if (arrived == p.k_split - 1) {
                    __threadfence();
#pragma unroll
                    for (int q = 0; q < P; ++q) {
                        const int t0 = q * W + ch * HALF;
                        if (n < p.M) {
                            const int32_t* src = p.partial + static_cast<int64_t>(t0) * p.M + n;
#pragma unroll
                            for (int t = 0; t < HALF; ++t) {
                                if (t0 + t < p.N) acc[q][t] = __ldcg(src);
                                src += p.M;
                            }
                        }
                        s8w_store<EPI, HALF>(acc[q], p, n, t0, sxs, swn, bn);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}


// Whether each kernel instance (epilogue x token tile) has its shared-memory
// attribute set, per device: four narrow and six wide token tiles per epilogue.
bool g_configured[64][20];

// Int8-operand GEMM plan for a weight matrix of N rows and K columns:
// weight tiles, stages of stage_k K (128 up to 96 tokens, 64 beyond), and
// the K split (1: none), each split at least 256 K.  K is split only when the
// weight tiles alone leave most SMs idle; the split count comes from the SM
// count, the need for the split buffers only from the shape.
struct S8Plan {
    int num_m, k_stages, k_split, split_stages;
};

constexpr int S8_COUNTERS_PER_TILE = 8;  // one per 32-row group (and column half, beyond 96 tokens)

bool s8_split_possible(int64_t N, int64_t K) {
    return (N + BM - 1) / BM <= S8_SPLIT_MAX_TILES && (K + S8_BK - 1) / S8_BK >= 4;
}

S8Plan s8_plan(int64_t N, int64_t K, int num_sms, int stage_k) {
    S8Plan pl;
    pl.num_m = static_cast<int>((N + BM - 1) / BM);
    pl.k_stages = static_cast<int>((K + stage_k - 1) / stage_k);
    int s = 1;
    if (s8_split_possible(N, K)) {
        s = num_sms / pl.num_m;
        if (s > S8_SPLIT_MAX) s = S8_SPLIT_MAX;
        if (s > pl.k_stages / (256 / stage_k)) s = pl.k_stages / (256 / stage_k);
        if (s < 2) s = 1;
    }
    pl.split_stages = (pl.k_stages + s - 1) / s;  // no split is left empty
    pl.k_split = (pl.k_stages + pl.split_stages - 1) / pl.split_stages;
    return pl;
}

size_t s8_align(size_t v) { return (v + 255) & ~size_t(255); }

// One launch of kernel k (instance id of g_configured) with SMEM bytes of
// dynamic shared memory, THREADS threads and one CTA per work unit (at most
// one per SM), after the tokens' image is written.
template <typename Kernel>
cudaError_t launch_s8_kernel(Kernel k, int id, size_t smem, int threads, const CUtensorMap& tmA,
                             const CUtensorMap& tmB, const S8Params& p, int ctas, cudaStream_t st) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!g_configured[dev][id]) {
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        g_configured[dev][id] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, tmA, tmB, p);
}

template <int EPI, int BN>
cudaError_t launch_s8_bn(const CUtensorMap& tmA, const CUtensorMap& tmB, const S8Params& p, int ctas,
                         cudaStream_t st) {
    constexpr int id = (EPI == kEpiPostscaleS32 ? 10 : 0) + (BN == 16 ? 0 : BN == 32 ? 1 : BN == 64 ? 2 : 3);
    static_assert(BN == 16 || BN == 32 || BN == 64 || BN == 96, "narrow token tile");
    return launch_s8_kernel(gemm_s8_kernel<EPI, BN>, id, CfgS8<BN>::SMEM, S8_THREADS, tmA, tmB, p, ctas, st);
}

template <int EPI, int BN>
cudaError_t launch_s8w_bn(const CUtensorMap& tmA, const CUtensorMap& tmB, const S8Params& p, int ctas,
                          cudaStream_t st) {
    constexpr int id = (EPI == kEpiPostscaleS32 ? 10 : 0) + 4 + (BN - 128) / 32;
    static_assert(BN >= 128 && BN <= 288 && BN % 32 == 0, "wide token tile");
    return launch_s8_kernel(gemm_s8w_kernel<EPI, BN>, id, CfgS8W<BN>::SMEM, S8W_THREADS, tmA, tmB, p, ctas, st);
}

constexpr int S8_NARROW_MAX_TOKENS = 96;  // gemm_s8_kernel up to this many tokens, gemm_s8w_kernel beyond

// Token tile of the int8-operand GEMM for T tokens: the narrowest that holds
// them (16 .. 96 on the narrow kernel, 128 .. 288 in steps of 32 on the wide one).
int s8_token_tile(int64_t T) {
    if (T <= S8_NARROW_MAX_TOKENS) return T <= 16 ? 16 : T <= 32 ? 32 : T <= 64 ? 64 : 96;
    return static_cast<int>((T + 31) / 32 * 32);
}

// The GEMM on int8 operands (M <= 288 tokens): s8_prep_kernel, then
// gemm_s8_kernel (up to 96 tokens) or gemm_s8w_kernel with one CTA per work
// unit (at most one per SM).  a.partial is the scratch of
// s8_workspace_bytes(M, N, K): the tokens' fp16 image, then (when K may be
// split) the int32 sums [M][N] and the arrival counters.
template <int EPI>
cudaError_t launch_s8(const void* Xq, const void* Wq, const GemmArgs& a, int num_sms,
                      PFN_cuTensorMapEncodeTiled_v12000 encode, cudaStream_t st, char* detail, size_t n) {
    const int64_t T = a.M, N = a.N, K = a.K;
    const bool wide = T > S8_NARROW_MAX_TOKENS;
    const int stage_k = wide ? S8W_BK : S8_BK;
    const S8Plan pl = s8_plan(N, K, num_sms, stage_k);
    uint8_t* ws = reinterpret_cast<uint8_t*>(a.partial);
    const size_t img_bytes = s8_align(static_cast<size_t>(T) * K * 2);
    const size_t sum_bytes = s8_align(static_cast<size_t>(T) * N * 4);
    const size_t cnt_bytes = s8_align(static_cast<size_t>(pl.num_m) * S8_COUNTERS_PER_TILE * 4);

    CUtensorMap tmA, tmB;
    {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
        cuuint32_t box[2] = {static_cast<cuuint32_t>(stage_k), static_cast<cuuint32_t>(BM)};
        cuuint32_t estr[2] = {1, 1};
        CUresult r = encode(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(Wq), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE,
                            wide ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            snprintf(detail, n, "cuTensorMapEncodeTiled(weight codes: %lld x %lld) returned %d", (long long)N,
                     (long long)K, (int)r);
            return cudaErrorInvalidValue;
        }
    }
    const int bn = s8_token_tile(T);
    {
        // the narrow kernel loads all bn token rows per box, the wide one each part
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(T)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
        cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(wide ? bn / s8w_parts(bn) : bn)};
        cuuint32_t estr[2] = {1, 1};
        CUresult r = encode(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, ws, dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            snprintf(detail, n, "cuTensorMapEncodeTiled(token image: %lld x %lld) returned %d", (long long)T,
                     (long long)K, (int)r);
            return cudaErrorInvalidValue;
        }
    }

    // the token image, and zeroed sums and counters for a split K (unless the
    // kernel before this one wrote them)
    const int64_t n16 = a.tokens_widened ? 0 : T * K / 16;
    const int64_t nz16 = pl.k_split > 1 ? static_cast<int64_t>((sum_bytes + cnt_bytes) / 16) : 0;
    int64_t grid = ((n16 > nz16 ? n16 : nz16) + 255) / 256;
    if (grid > static_cast<int64_t>(num_sms) * 4) grid = static_cast<int64_t>(num_sms) * 4;
    if (grid < 1) grid = 1;
    if (!a.tokens_widened) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(256);
        cfg.stream = st;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, s8_prep_kernel, static_cast<const uint4*>(Xq), n16,
                                           reinterpret_cast<uint4*>(ws), reinterpret_cast<uint4*>(ws + img_bytes),
                                           nz16);
        if (e != cudaSuccess) return e;
    }

    S8Params p{};
    p.sx = a.sx;
    p.sw = a.sw;
    p.bias = static_cast<const uint16_t*>(a.bias);
    p.out = a.out;
    p.M = static_cast<int>(N);  // kernel rows: weight rows
    p.N = static_cast<int>(T);  // kernel columns: tokens
    p.K = static_cast<int>(K);
    p.num_m = pl.num_m;
    p.k_stages = pl.k_stages;
    p.k_split = pl.k_split;
    p.split_stages = pl.split_stages;
    p.num_tiles = pl.num_m * pl.k_split;
    p.partial = pl.k_split > 1 ? reinterpret_cast<int32_t*>(ws + img_bytes) : nullptr;
    p.counters = pl.k_split > 1 ? reinterpret_cast<int32_t*>(ws + img_bytes + sum_bytes) : nullptr;
    p.a_settled = a.weights_settled ? 1 : 0;
    const int ctas = p.num_tiles < num_sms ? p.num_tiles : num_sms;
    switch (bn) {
        case 16: return launch_s8_bn<EPI, 16>(tmA, tmB, p, ctas, st);
        case 32: return launch_s8_bn<EPI, 32>(tmA, tmB, p, ctas, st);
        case 64: return launch_s8_bn<EPI, 64>(tmA, tmB, p, ctas, st);
        case 96: return launch_s8_bn<EPI, 96>(tmA, tmB, p, ctas, st);
        case 128: return launch_s8w_bn<EPI, 128>(tmA, tmB, p, ctas, st);
        case 160: return launch_s8w_bn<EPI, 160>(tmA, tmB, p, ctas, st);
        case 192: return launch_s8w_bn<EPI, 192>(tmA, tmB, p, ctas, st);
        case 224: return launch_s8w_bn<EPI, 224>(tmA, tmB, p, ctas, st);
        case 256: return launch_s8w_bn<EPI, 256>(tmA, tmB, p, ctas, st);
        case 288: return launch_s8w_bn<EPI, 288>(tmA, tmB, p, ctas, st);
        default:
            snprintf(detail, n, "int8-operand GEMM: %lld tokens exceed the widest token tile", (long long)T);
            return cudaErrorInvalidValue;
    }
}


}  // namespace

void s8_scratch_zero(int64_t M, int64_t N, int64_t K, int num_sms, size_t* offset, size_t* bytes) {
    const S8Plan pl = s8_plan(N, K, num_sms, M > S8_NARROW_MAX_TOKENS ? S8W_BK : S8_BK);
    *offset = s8_align(static_cast<size_t>(M) * K * 2);
    *bytes = pl.k_split > 1 ? s8_align(static_cast<size_t>(M) * N * 4) +
                                  s8_align(static_cast<size_t>(pl.num_m) * S8_COUNTERS_PER_TILE * 4)
                            : 0;
}

size_t s8_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    size_t b = s8_align(static_cast<size_t>(M) * K * 2);
    if (s8_split_possible(N, K))
        b += s8_align(static_cast<size_t>(M) * N * 4) +
             s8_align(static_cast<size_t>((N + BM - 1) / BM) * S8_COUNTERS_PER_TILE * 4);
    return b;
}

cudaError_t launch_gemm_s8(int epilogue, const void* Xq, const void* Wq, const GemmArgs& a, int num_sms,
                          void* encode_fn, cudaStream_t st, char* detail, size_t n) {
    if (n) detail[0] = 0;
    if (!a.partial) {
        snprintf(detail, n, "int8-operand GEMM without its scratch");
        return cudaErrorInvalidValue;
    }
    auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(encode_fn);
    cudaError_t e;
    if (epilogue == kEpiPostscaleS32)
        e = launch_s8<kEpiPostscaleS32>(Xq, Wq, a, num_sms, encode, st, detail, n);
    else if (epilogue == kEpiPostscaleBf16)
        e = launch_s8<kEpiPostscaleBf16>(Xq, Wq, a, num_sms, encode, st, detail, n);
    else
        e = cudaErrorInvalidValue;
    if (e != cudaSuccess && n && detail[0] == 0)
        snprintf(detail, n, "int8-operand GEMM launch: %s", cudaGetErrorString(e));
    return e;
}

cudaError_t gemm_s8_read_device_error(unsigned int* code) {
    unsigned int v = 0, z = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof v);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbol(g_device_error, &z, sizeof z);
    *code = v;
    return e;
}

}  // namespace w8a8
