// Stage S1 (route metadata), S2 (dispatch gather) and S6 (combine), plus the bounded-wait
// test hook.
//
// Route metadata follows the count -> prefix sum -> scatter scheme of the layout-metadata
// page (§1, §3.2-3.5): every CTA counts its ids per expert in shared memory with
// warp-aggregated atomics, claims a contiguous range of each expert's rows with one global
// atomicAdd per (CTA, expert) -- the returned old value is the CTA's base -- and a second
// kernel scans the final counts into offsets. Unlike the prior art's single persistent
// kernel with a grid barrier, the scan runs as its own tiny launch, so no CTA ever waits on
// another.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kRouteThreads = 256;
constexpr int kRouteItems = 4;                        // ids per thread in the count kernel
constexpr int kRouteChunk = kRouteThreads * kRouteItems;

// Expert of slot i = t*Kt + k of the plan: the caller's id for the Kr routed slots; shared
// expert Er + (k - Kr) for the slots after them (DeepGEMM page §6: a shared expert takes every
// token, in the combine slot after the routed ones). A routed id that names a shared expert is
// returned as Et = Er + (Kt - Kr), out of range, so that it counts as a bad route.
__device__ __forceinline__ int route_id(const int32_t* __restrict__ ids, int i, int Kt, int Kr, int Er) {
    if (Kt == Kr) return ids[i];
    const int t = i / Kt, k = i - t * Kt;
    if (k >= Kr) return Er + (k - Kr);
    const int e = ids[t * Kr + k];
    return e >= Er ? Er + (Kt - Kr) : e;
}

// Count ids per expert in shared memory (warp-aggregated), claim each expert's range with a
// global atomicAdd and record every id's position inside its expert.
__global__ void __launch_bounds__(kRouteThreads) route_count_claim_kernel(const int32_t* __restrict__ ids, int n_ids,
                                                                          int Kt, int Kr, int Er,
                                                                          int E, int32_t* __restrict__ claim,
                                                                          int32_t* __restrict__ pos,
                                                                          int32_t* __restrict__ hdr) {
    extern __shared__ int32_t smem[];
    int32_t* hist = smem;      // [E] ids of this CTA per expert
    int32_t* base = smem + E;  // [E] this CTA's first position in each expert
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int begin = blockIdx.x * kRouteChunk;
    int expert[kRouteItems];
    int rank[kRouteItems];
#pragma unroll
    for (int j = 0; j < kRouteItems; ++j) {
        const int i = begin + j * kRouteThreads + threadIdx.x;
        const bool in = i < n_ids;
        int e = in ? route_id(ids, i, Kt, Kr, Er) : -1;
        const bool valid = in && e >= 0 && e < E;
        if (in && !valid && e != -1) record_error(hdr, MOE_ERR_BAD_ROUTE);
        expert[j] = valid ? e : -1;
        rank[j] = -1;
        const unsigned active = __ballot_sync(0xffffffffu, valid);
        if (valid) {
            const unsigned peers = __match_any_sync(active, e);   // lanes routed to the same expert
            const int leader = __ffs(peers) - 1;
            int b = 0;
            if (lane == leader) b = atomicAdd(&hist[e], __popc(peers));
            b = __shfl_sync(peers, b, leader);
            rank[j] = b + __popc(peers & ((1u << lane) - 1u));
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int c = hist[e];
        base[e] = c ? atomicAdd(&claim[e], c) : 0;               // global offset claim
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kRouteItems; ++j) {
        const int i = begin + j * kRouteThreads + threadIdx.x;
        if (i < n_ids) pos[i] = expert[j] >= 0 ? base[expert[j]] + rank[j] : -1;
    }
}

// Exclusive scan over up to 1024 values, one per thread of a 1024-thread block.
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
        int s = w;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, s, d);
            if (lane >= d) s += y;
        }
        warp_sums[lane] = s - w;  // exclusive prefix of the warp totals
        if (lane == 31) *total = s;
    }
    __syncthreads();
    const int out = x - v + warp_sums[warp];
    __syncthreads();
    return out;
}

// counts -> offsets, padded offsets and tile offsets (the padding rows of the pools keep the -1
// that launch_route writes into pool_src before the scatter).
__global__ void __launch_bounds__(1024) route_scan_kernel(int E, const int32_t* __restrict__ claim,
                                                          int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ pad_off, int32_t* __restrict__ tile_off,
                                                          int32_t* __restrict__ pool_src, int32_t* __restrict__ hdr,
                                                          int32_t* __restrict__ counts_out,
                                                          int32_t* __restrict__ offsets_out) {
    __shared__ int warp_sums[32];
    __shared__ int total_rows, total_tiles;
    const int e = threadIdx.x;
    const int c = e < E ? claim[e] : 0;
    const int tiles = (c + kTileRows - 1) / kTileRows;
    const int off = block_exclusive_scan(c, warp_sums, &total_rows);
    const int toff = block_exclusive_scan(tiles, warp_sums, &total_tiles);
    if (e < E) {
        counts[e] = c;
        offsets[e] = off;
        tile_off[e] = toff;
        pad_off[e] = toff * kTileRows;
        if (counts_out) counts_out[e] = c;
        if (offsets_out) offsets_out[e] = off;
    }
    if (e == 0) {
        offsets[E] = total_rows;
        tile_off[E] = total_tiles;
        pad_off[E] = total_tiles * kTileRows;
        if (offsets_out) offsets_out[E] = total_rows;
        hdr[kHdrRows] = total_rows;
        hdr[kHdrPadRows] = total_tiles * kTileRows;
        hdr[kHdrTiles] = total_tiles;
    }
}

// S1 in one CTA for up to kSmallIds ids and 1024 experts (decode steps): the same count
// (warp-aggregated shared-memory atomics), scan and scatter as the three kernels above, with every
// id's expert and rank kept in registers between the phases, so one launch replaces three. Measured:
// the decode step (1024 ids) 9 us shorter; with 8192-12288 ids the one CTA's atomics (a few experts
// take many ids) made the step slower than the multi-CTA count, hence the bound.
constexpr int kSmallThreads = 1024, kSmallItems = 4, kSmallIds = kSmallThreads * kSmallItems;
__global__ void __launch_bounds__(kSmallThreads) route_small_kernel(const int32_t* __restrict__ ids, int n_ids, int Kt,
                                                                   int Kr, int Er, int E, int32_t* __restrict__ counts,
                                                                   int32_t* __restrict__ offsets,
                                                                   int32_t* __restrict__ pad_off,
                                                                   int32_t* __restrict__ tile_off,
                                                                   int32_t* __restrict__ row_src,
                                                                   int32_t* __restrict__ pool_src,
                                                                   int32_t* __restrict__ slot_row,
                                                                   int32_t* __restrict__ hdr,
                                                                   int32_t* __restrict__ counts_out,
                                                                   int32_t* __restrict__ offsets_out,
                                                                   int32_t* __restrict__ row_src_out, int64_t pool_rows) {
    __shared__ int hist[1024];   // ids per expert, then (after the scan) each expert's first row
    __shared__ int pad_s[1024];  // each expert's first padded pool row
    __shared__ int warp_sums[32];
    __shared__ int total_rows, total_tiles;
    const int lane = threadIdx.x & 31;
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    int expert[kSmallItems];
    int rank[kSmallItems];
#pragma unroll
    for (int j = 0; j < kSmallItems; ++j) {
        const int i = j * kSmallThreads + threadIdx.x;
        const bool in = i < n_ids;
        const int e = in ? route_id(ids, i, Kt, Kr, Er) : -1;
        const bool valid = in && e >= 0 && e < E;
        if (in && !valid && e != -1) record_error(hdr, MOE_ERR_BAD_ROUTE);
        expert[j] = valid ? e : -1;
        rank[j] = -1;
        const unsigned active = __ballot_sync(0xffffffffu, valid);
        if (valid) {
            const unsigned peers = __match_any_sync(active, e);  // lanes routed to the same expert
            const int leader = __ffs(peers) - 1;
            int b = 0;
            if (lane == leader) b = atomicAdd(&hist[e], __popc(peers));
            b = __shfl_sync(peers, b, leader);
            rank[j] = b + __popc(peers & ((1u << lane) - 1u));
        }
    }
    __syncthreads();
    // counts -> offsets, padded offsets and tile offsets (one expert per thread)
    const int me = threadIdx.x;
    const int c = me < E ? hist[me] : 0;
    const int off = block_exclusive_scan(c, warp_sums, &total_rows);
    const int toff = block_exclusive_scan((c + kTileRows - 1) / kTileRows, warp_sums, &total_tiles);
    if (me < E) {
        counts[me] = c;
        offsets[me] = off;
        tile_off[me] = toff;
        pad_off[me] = toff * kTileRows;
        hist[me] = off;
        pad_s[me] = toff * kTileRows;
        if (counts_out) counts_out[me] = c;
        if (offsets_out) offsets_out[me] = off;
    }
    if (me == 0) {
        offsets[E] = total_rows;
        tile_off[E] = total_tiles;
        pad_off[E] = total_tiles * kTileRows;
        if (offsets_out) offsets_out[E] = total_rows;
        hdr[kHdrRows] = total_rows;
        hdr[kHdrPadRows] = total_tiles * kTileRows;
        hdr[kHdrTiles] = total_tiles;
    }
    __syncthreads();
    // scatter, both directions of the identity map
#pragma unroll
    for (int j = 0; j < kSmallItems; ++j) {
        const int i = j * kSmallThreads + threadIdx.x;
        if (i >= n_ids) continue;
        const int e = expert[j];
        if (e < 0) {
            slot_row[i] = -1;
            continue;
        }
        const int row = hist[e] + rank[j];
        const int prow = pad_s[e] + rank[j];
        if (!debug_ok(hdr, row >= 0 && row < n_ids && prow >= 0 && prow < pool_rows)) {
            slot_row[i] = -1;
            continue;
        }
        row_src[row] = i;
        if (row_src_out) row_src_out[row] = i;
        pool_src[prow] = i;
        slot_row[i] = prow;
    }
}

// Scatter every routed (i,k) to its pool row and record both directions of the identity map.
__global__ void route_scatter_kernel(const int32_t* __restrict__ ids, int n_ids, int Kt, int Kr, int Er, int E,
                                     const int32_t* __restrict__ pos,
                                     const int32_t* __restrict__ offsets, const int32_t* __restrict__ pad_off,
                                     int32_t* __restrict__ row_src, int32_t* __restrict__ pool_src,
                                     int32_t* __restrict__ slot_row, int32_t* __restrict__ row_src_out,
                                     int32_t* __restrict__ hdr, int64_t pool_rows) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n_ids) return;
    const int e = route_id(ids, i, Kt, Kr, Er);
    const int p = pos[i];
    if (e < 0 || e >= E || p < 0) {
        slot_row[i] = -1;
        return;
    }
    const int row = offsets[e] + p;
    const int prow = pad_off[e] + p;
    if (!debug_ok(hdr, row >= 0 && row < n_ids && prow >= 0 && prow < pool_rows)) {
        slot_row[i] = -1;
        return;
    }
    row_src[row] = i;
    if (row_src_out) row_src_out[row] = i;
    pool_src[prow] = i;
    slot_row[i] = prow;
}

// S2: copy x row (token = i / K) and its scale row into the pool row of every routed slot i
// (slot_row; -1 for a masked route). Iterating the slots rather than the pool rows skips the
// padding rows without reading them (at decode sizes most pool rows are padding). Padding rows are
// left as they are: every consumer computes rows (tokens) independently and drops their results.
__global__ void __launch_bounds__(128) dispatch_gather_kernel(const uint4* __restrict__ x, const uint32_t* __restrict__ xs,
                                                              const int32_t* __restrict__ slot_row,
                                                              int32_t* __restrict__ hdr, int K, int row_vecs,
                                                              int scale_words, uint4* __restrict__ xp,
                                                              uint32_t* __restrict__ xps, int64_t n_ids,
                                                              int64_t pool_rows) {
    for (int64_t i = blockIdx.x; i < n_ids; i += gridDim.x) {
        const int r = debug_row(hdr, slot_row[i], pool_rows);
        if (r < 0) continue;  // masked route
        const int64_t src = i;
        uint4* dst = xp + (size_t)r * row_vecs;
        const uint4* s = x + (size_t)(src / K) * row_vecs;
        for (int v = threadIdx.x; v < row_vecs; v += blockDim.x) dst[v] = s[v];
        for (int w = threadIdx.x; w < scale_words; w += blockDim.x)
            xps[(size_t)r * scale_words + w] = xs[(size_t)(src / K) * scale_words + w];
    }
}

// S2 for the quantised modes: copies the codes and scale rows like dispatch_gather_kernel. For
// the INT8 mode it also writes the codes as two f16 planes, hi = floor(q/16) and lo = q mod 16
// (q = 16*hi + lo, both exact in f16), the operand of the INT8 tensor-core GEMM: with them every
// fp32 partial sum of that GEMM stays an exactly representable integer. For A8W4-INT the plane
// is the codes themselves as f16 (int8 x int4 products are small enough without the split), in
// the order of w4_plane_pos, and the row's code sum goes to `sums`.
// Each thread keeps four 16-byte loads in flight before its stores, and the next slot's pool row
// is read while the current row is copied (a row costs two dependent loads otherwise). Like
// dispatch_gather_kernel it iterates the routed slots (slot_row), so padding rows cost nothing.
template <int MODE>
__global__ void __launch_bounds__(128) dispatch_gather_q_kernel(const uint8_t* __restrict__ x, const uint8_t* __restrict__ xs,
                                                                const int32_t* __restrict__ slot_row,
                                                                int32_t* __restrict__ hdr, int K, int H,
                                                                int scale_bytes, int64_t pool_rows, uint8_t* __restrict__ xp,
                                                                uint8_t* __restrict__ xps, uint16_t* __restrict__ xb,
                                                                int32_t* __restrict__ sums, int64_t n_ids) {
    constexpr int kUnroll = 4;
    __shared__ int red[4];
    const int nv = H / 16;                 // 16-byte vectors of a row of codes
    const int scale_words = scale_bytes / 4;
    int64_t i = blockIdx.x;
    int r = i < n_ids ? debug_row(hdr, __ldg(slot_row + i), pool_rows) : -1;
    while (i < n_ids) {
        const int64_t in = i + gridDim.x;
        const int r_next = in < n_ids ? debug_row(hdr, __ldg(slot_row + in), pool_rows) : -1;
        if (r >= 0) {  // a masked route writes nothing; padding rows are left as they are
            const int64_t tok = i / K;
            const uint4* xs4 = reinterpret_cast<const uint4*>(x + tok * H);
            uint4* xd = reinterpret_cast<uint4*>(xp + (int64_t)r * H);
            int row_sum = 0;  // A8W4-INT
            for (int v0 = threadIdx.x; v0 < nv; v0 += kUnroll * blockDim.x) {
                uint4 c[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int v = v0 + u * blockDim.x;
                    if (v < nv) c[u] = __ldg(xs4 + v);
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int v = v0 + u * blockDim.x;
                    if (v >= nv) break;
                    xd[v] = c[u];
                    if constexpr (MODE == MOE_A8W4_INT) {
                        const uint8_t* b = reinterpret_cast<const uint8_t*>(&c[u]);
                        uint32_t f[8];  // word 4g + j: codes 8g + j and 8g + 4 + j
#pragma unroll
                        for (int g = 0; g < 2; ++g)
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const int q0 = (int8_t)b[8 * g + j], q1 = (int8_t)b[8 * g + 4 + j];
                                f[4 * g + j] = (uint32_t)float_to_f16_bits((float)q0) |
                                               ((uint32_t)float_to_f16_bits((float)q1) << 16);
                                row_sum += q0 + q1;
                            }
                        uint4* d = reinterpret_cast<uint4*>(xb + (int64_t)r * H + v * 16);
                        d[0] = make_uint4(f[0], f[1], f[2], f[3]);
                        d[1] = make_uint4(f[4], f[5], f[6], f[7]);
                    } else if constexpr (MODE == MOE_A8W8_INT8) {
                        const uint8_t* b = reinterpret_cast<const uint8_t*>(&c[u]);
                        uint32_t hi[8], lo[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int q0 = (int8_t)b[2 * j], q1 = (int8_t)b[2 * j + 1];
                            hi[j] = (uint32_t)float_to_f16_bits((float)(q0 >> 4)) |
                                    ((uint32_t)float_to_f16_bits((float)(q1 >> 4)) << 16);
                            lo[j] = (uint32_t)float_to_f16_bits((float)(q0 & 15)) |
                                    ((uint32_t)float_to_f16_bits((float)(q1 & 15)) << 16);
                        }
                        uint4* dh = reinterpret_cast<uint4*>(xb + (int64_t)r * H + v * 16);
                        uint4* dl = reinterpret_cast<uint4*>(xb + (pool_rows + r) * H + v * 16);
                        dh[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        dh[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
                        dl[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                        dl[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
                    }
                }
            }
            for (int w = threadIdx.x; w < scale_words; w += blockDim.x) {
                const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(xs + tok * scale_bytes) + w);
                if constexpr (MODE == MOE_A8W4_FP8_FP4) {
                    // the block-scaled MMA takes the exponent byte as a UE8M0 scale, so the scale must be
                    // 2^e with -127 <= e <= 127: a positive normal fp32 with a zero mantissa, or 2^-127
                    // (the subnormal whose exponent byte is 0)
                    const uint32_t sexp = v >> 23;  // sign and exponent bits
                    const bool pow2 = (v & 0x7fffffu) == 0 ? (sexp >= 1 && sexp <= 254) : v == 0x00400000u;
                    if (!pow2) record_error(hdr, MOE_ERR_BAD_SCALE);
                }
                reinterpret_cast<uint32_t*>(xps + (int64_t)r * scale_bytes)[w] = v;
            }
            if constexpr (MODE == MOE_A8W4_INT) {  // r >= 0 is uniform across the block
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) row_sum += __shfl_xor_sync(0xffffffffu, row_sum, o);
                if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = row_sum;
                __syncthreads();
                if (threadIdx.x == 0) sums[r] = red[0] + red[1] + red[2] + red[3];
                __syncthreads();
            }
        }
        i = in;
        r = r_next;
    }
}

// S2 with the operator's own activation quantisation (Ascend page, A8W8-INT and A8W4-INT use
// cases "EP Dispatch": per token s = max|X[i,:]|/127, q = round(X/s); A8W8-FP use case: Q_MX with groups
// of 32 and E8M0 scales; FP8 activations x FP4 weights: the same shared-exponent rule on groups
// of 128, fp32 power-of-two scales, the mode's x format). One CTA per token: its bf16 row is
// quantised once and written to each of its K pool rows. Warp w takes 128-element chunks, 4
// elements per lane. Every code is decided on fp32 values: IEEE division for the int8 scale
// and quotient, exact power-of-two scaling before the e4m3 rounding.
template <int MODE>
__global__ void __launch_bounds__(256) dispatch_quant_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ slot_row,
                                                             int T, int K, int H, int64_t pool_rows, uint8_t* __restrict__ xp,
                                                             uint8_t* __restrict__ xps, uint16_t* __restrict__ xb,
                                                             int32_t* __restrict__ sums, int32_t* __restrict__ hdr) {
    __shared__ float red[8];
    __shared__ int red_sum[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        // pool row of slot `lane` (K <= 32), shuffled to all lanes when the chunk is stored
        const int my_row = lane < K ? debug_row(hdr, __ldg(slot_row + (int64_t)t * K + lane), pool_rows) : -1;
        const uint2* xr = reinterpret_cast<const uint2*>(x + (int64_t)t * H);  // 4 bf16 per uint2
        float s_int8 = 0.0f;
        if constexpr (int_mode(MODE)) {
            float m = 0.0f;
            for (int c = threadIdx.x; c < H / 4; c += blockDim.x) {
                const uint2 v = __ldg(xr + c);
                m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16_bits_to_float(v.x & 0xffff)), fabsf(bf16_bits_to_float(v.x >> 16))),
                                   fmaxf(fabsf(bf16_bits_to_float(v.y & 0xffff)), fabsf(bf16_bits_to_float(v.y >> 16)))));
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane == 0) red[warp] = m;
            __syncthreads();
            float amax = red[0];
#pragma unroll
            for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
            __syncthreads();
            s_int8 = fmaxf(__fdiv_rn(amax, 127.0f), 1e-8f);
        }
        int code_sum = 0;  // A8W4-INT
        for (int c0 = warp * 128; c0 < H; c0 += 8 * 128) {
            const uint2 v = __ldg(xr + c0 / 4 + lane);
            const float f[4] = {bf16_bits_to_float(v.x & 0xffff), bf16_bits_to_float(v.x >> 16),
                                bf16_bits_to_float(v.y & 0xffff), bf16_bits_to_float(v.y >> 16)};
            uint32_t code = 0, hi[2] = {0, 0}, lo[2] = {0, 0};
            int ex = 0;  // FP8 modes: exponent of this lane's group
            if constexpr (int_mode(MODE)) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float q = rintf(__fdiv_rn(f[c], s_int8));
                    q = fminf(fmaxf(q, -127.0f), 127.0f);
                    const int qi = (int)q;
                    code |= (uint32_t)(qi & 0xff) << (8 * c);
                    if constexpr (MODE == MOE_A8W8_INT8) {
                        hi[c >> 1] |= (uint32_t)float_to_f16_bits((float)(qi >> 4)) << (16 * (c & 1));
                        lo[c >> 1] |= (uint32_t)float_to_f16_bits((float)(qi & 15)) << (16 * (c & 1));
                    } else {  // A8W4-INT: the codes as one f16 plane (order below)
                        hi[c >> 1] |= (uint32_t)float_to_f16_bits((float)qi) << (16 * (c & 1));
                        code_sum += qi;
                    }
                }
                if constexpr (MODE == MOE_A8W4_INT) {
                    // codes 0-3 of a group of 8 are in an even lane, 4-7 in the next one; the plane
                    // holds q0 q4 q1 q5 (even lane) and q2 q6 q3 q7 (odd lane)
                    const bool odd = lane & 1;
                    const uint32_t got = __shfl_xor_sync(0xffffffffu, odd ? hi[0] : hi[1], 1);
                    const uint32_t mine = odd ? hi[1] : hi[0];
                    hi[0] = odd ? (got & 0xffffu) | (mine << 16) : (mine & 0xffffu) | (got << 16);
                    hi[1] = odd ? (got >> 16) | (mine & 0xffff0000u) : (mine >> 16) | (got & 0xffff0000u);
                }
            } else {
                float m = fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3])));
                // group of 32 = 8 lanes (A8W8-FP8) or of 128 = the warp (FP8 x FP4)
                constexpr int kLanes = MODE == MOE_A8W4_FP8_FP4 ? 32 : 8;
                constexpr bool kE5 = MODE == MOE_A8W8_FP8_E5M2;
#pragma unroll
                for (int o = 1; o < kLanes; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                ex = mx_exponent_fp8<kE5>(m);
                const float inv = exp2_neg_int(ex);
#pragma unroll
                for (int c = 0; c < 4; ++c) code |= (uint32_t)float_to_fp8_satfinite<kE5>(f[c] * inv) << (8 * c);
            }
            for (int k = 0; k < K; ++k) {
                const int prow = __shfl_sync(0xffffffffu, my_row, k);
                if (prow < 0) continue;  // masked route (uniform across the warp)
                reinterpret_cast<uint32_t*>(xp + (int64_t)prow * H + c0)[lane] = code;
                if constexpr (MODE == MOE_A8W8_INT8) {
                    reinterpret_cast<uint2*>(xb + (int64_t)prow * H + c0)[lane] = make_uint2(hi[0], hi[1]);
                    reinterpret_cast<uint2*>(xb + (pool_rows + prow) * H + c0)[lane] = make_uint2(lo[0], lo[1]);
                } else if constexpr (MODE == MOE_A8W4_INT) {
                    reinterpret_cast<uint2*>(xb + (int64_t)prow * H + c0)[lane] = make_uint2(hi[0], hi[1]);
                } else if constexpr (MODE == MOE_A8W8_FP8 || MODE == MOE_A8W8_FP8_E5M2) {
                    if ((lane & 7) == 0) xps[(int64_t)prow * (H / 32) + c0 / 32 + lane / 8] = (uint8_t)(ex + 127);
                } else {
                    // 2^ex as fp32 (2^-127, a subnormal, for an all-zero group)
                    if (lane == 0) reinterpret_cast<float*>(xps)[(int64_t)prow * (H / 128) + c0 / 128] = ue8m0_to_float((uint8_t)(ex + 127));
                }
            }
        }
        if constexpr (MODE == MOE_A8W4_INT) {
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) code_sum += __shfl_xor_sync(0xffffffffu, code_sum, o);
            if (lane == 0) red_sum[warp] = code_sum;
            __syncthreads();
            code_sum = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) code_sum += red_sum[w];
            __syncthreads();
        }
        if constexpr (int_mode(MODE)) {
            if (threadIdx.x < K) {
                const int prow = my_row;
                if (prow >= 0) {
                    reinterpret_cast<float*>(xps)[prow] = s_int8;
                    if constexpr (MODE == MOE_A8W4_INT) sums[prow] = code_sum;
                }
            }
        }
    }
}

// S6: y[t, 8j..8j+7] = bf16( sum_k comb[t*K+k, 8j..8j+7] ), fp32 sum in slot order. The slots are
// read eight at a time, all loads in flight before the first add (a masked slot's row is read, it
// lies inside comb, and skipped), so a thread waits for one memory round trip per eight slots.
__global__ void __launch_bounds__(256) combine_kernel(const uint4* __restrict__ comb, const int32_t* __restrict__ slot_row,
                                                      int T, int K, int row_vecs, uint4* __restrict__ y) {
    constexpr int kSlots = 8;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)T * row_vecs) return;
    const int t = (int)(idx / row_vecs);
    const int v = (int)(idx % row_vecs);
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    for (int k0 = 0; k0 < K; k0 += kSlots) {
        uint4 c[kSlots];
        int r[kSlots];
#pragma unroll
        for (int u = 0; u < kSlots; ++u) {
            const int k = k0 + u;
            r[u] = k < K ? __ldg(slot_row + t * K + k) : -1;
            if (k < K) c[u] = __ldg(comb + ((size_t)t * K + k) * row_vecs + v);
        }
#pragma unroll
        for (int u = 0; u < kSlots; ++u) {
            if (r[u] < 0) continue;  // masked route (or past K): contributes nothing
            const uint32_t w[4] = {c[u].x, c[u].y, c[u].z, c[u].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc[2 * j] = __fadd_rn(acc[2 * j], __uint_as_float(w[j] << 16));
                acc[2 * j + 1] = __fadd_rn(acc[2 * j + 1], __uint_as_float(w[j] & 0xffff0000u));
            }
        }
    }
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        o[j] = (uint32_t)float_to_bf16_bits(acc[2 * j]) | ((uint32_t)float_to_bf16_bits(acc[2 * j + 1]) << 16);
    y[(size_t)t * row_vecs + v] = make_uint4(o[0], o[1], o[2], o[3]);
}

// Gates of the plan's slots with shared experts: the caller's [T, Kr] gates, then 1 for each of
// the Kt - Kr shared slots of a token.
__global__ void expand_gates_kernel(const float* __restrict__ g, int n, int Kt, int Kr, float* __restrict__ out) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int t = i / Kt, k = i - t * Kt;
    out[i] = k < Kr ? g[t * Kr + k] : 1.0f;
}

// Waits for hdr[kHdrWaitFlag] to become non-zero, at most timeout_ns; on time-out records
// MOE_ERR_TIMEOUT and returns.
__global__ void debug_wait_kernel(int32_t* hdr, uint64_t timeout_ns) {
    const uint64_t t0 = globaltimer_ns();
    volatile int32_t* flag = hdr + kHdrWaitFlag;
    while (*flag == 0) {
        if (globaltimer_ns() - t0 > timeout_ns) {
            record_error(hdr, MOE_ERR_TIMEOUT);
            return;
        }
        __nanosleep(1000);
    }
}

}  // namespace

cudaError_t launch_route(const Plan& p, const int32_t* topk_ids, int32_t* counts_out, int32_t* offsets_out,
                         int32_t* row_src_out, cudaStream_t s) {
    const int n_ids = p.T * p.K;
    // the header (error word, totals) and the per-expert claim counters are contiguous
    const size_t clear = reinterpret_cast<const uint8_t*>(p.claim + p.E) - reinterpret_cast<const uint8_t*>(p.hdr);
    cudaError_t e = cudaMemsetAsync(p.hdr, 0, clear, s);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(p.pool_src, 0xff, sizeof(int32_t) * (size_t)p.pool_rows, s);  // -1: padding row
    if (e != cudaSuccess) return e;
    if (n_ids <= kSmallIds && p.E <= kSmallThreads) {  // one launch for the whole stage
        route_small_kernel<<<1, kSmallThreads, 0, s>>>(topk_ids, n_ids, p.K, p.Kr, p.Er, p.E, p.counts, p.offsets,
                                                       p.pad_off, p.tile_off, p.row_src, p.pool_src, p.slot_row, p.hdr,
                                                       counts_out, offsets_out, row_src_out, p.pool_rows);
        return cudaGetLastError();
    }
    if (n_ids > 0) {
        const int blocks = (n_ids + kRouteChunk - 1) / kRouteChunk;
        route_count_claim_kernel<<<blocks, kRouteThreads, 2 * p.E * sizeof(int32_t), s>>>(
            topk_ids, n_ids, p.K, p.Kr, p.Er, p.E, p.claim, p.pos, p.hdr);
    }
    route_scan_kernel<<<1, 1024, 0, s>>>(p.E, p.claim, p.counts, p.offsets, p.pad_off, p.tile_off, p.pool_src, p.hdr,
                                         counts_out, offsets_out);
    if (n_ids > 0) {
        route_scatter_kernel<<<(n_ids + 255) / 256, 256, 0, s>>>(topk_ids, n_ids, p.K, p.Kr, p.Er, p.E, p.pos,
                                                                 p.offsets, p.pad_off, p.row_src, p.pool_src,
                                                                 p.slot_row, row_src_out, p.hdr, p.pool_rows);
    }
    return cudaGetLastError();
}

template <int MODE>
static cudaError_t dispatch_q(const Plan& p, const void* x, const void* x_scale, cudaStream_t s) {
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((int64_t)p.T * p.K, 152 * 16));
    dispatch_gather_q_kernel<MODE><<<grid, 128, 0, s>>>(static_cast<const uint8_t*>(x),
                                                        static_cast<const uint8_t*>(x_scale), p.slot_row, p.hdr, p.K,
                                                        p.H, (int)x_scale_row_bytes(MODE, p.H), p.pool_rows, p.x_pool,
                                                        p.x_pool_scale, p.x_planes, p.x_sums, (int64_t)p.T * p.K);
    return cudaGetLastError();
}

cudaError_t launch_dispatch(const Plan& p, const void* x, const void* x_scale, cudaStream_t s) {
    if (p.T == 0) return cudaSuccess;
    switch (p.mode) {
        case MOE_A8W8_FP8: return dispatch_q<MOE_A8W8_FP8>(p, x, x_scale, s);
        case MOE_A8W8_FP8_E5M2: return dispatch_q<MOE_A8W8_FP8_E5M2>(p, x, x_scale, s);
        case MOE_A8W8_INT8: return dispatch_q<MOE_A8W8_INT8>(p, x, x_scale, s);
        case MOE_A8W4_INT: return dispatch_q<MOE_A8W4_INT>(p, x, x_scale, s);
        case MOE_A8W4_FP8_FP4: return dispatch_q<MOE_A8W4_FP8_FP4>(p, x, x_scale, s);
        default: break;
    }
    const int row_vecs = p.H * x_elem_bytes(p.mode) / 16;
    const int scale_words = (int)(x_scale_row_bytes(p.mode, p.H) / 4);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((int64_t)p.T * p.K, 152 * 16));
    dispatch_gather_kernel<<<grid, 128, 0, s>>>(static_cast<const uint4*>(x), static_cast<const uint32_t*>(x_scale),
                                                p.slot_row, p.hdr, p.K, row_vecs, scale_words,
                                                reinterpret_cast<uint4*>(p.x_pool),
                                                reinterpret_cast<uint32_t*>(p.x_pool_scale), (int64_t)p.T * p.K,
                                                p.pool_rows);
    return cudaGetLastError();
}

cudaError_t launch_dispatch_quant(const Plan& p, const void* x_bf16, cudaStream_t s) {
    if (p.T == 0) return cudaSuccess;
    const int grid = (int)std::min<int64_t>(p.T, 152 * 8);
    const uint16_t* x = static_cast<const uint16_t*>(x_bf16);
    switch (p.mode) {
        case MOE_A8W8_FP8_E5M2:
            dispatch_quant_kernel<MOE_A8W8_FP8_E5M2><<<grid, 256, 0, s>>>(x, p.slot_row, p.T, p.K, p.H, p.pool_rows,
                                                                          p.x_pool, p.x_pool_scale, p.x_planes, p.x_sums, p.hdr);
            break;
        case MOE_A8W8_FP8:
            dispatch_quant_kernel<MOE_A8W8_FP8><<<grid, 256, 0, s>>>(x, p.slot_row, p.T, p.K, p.H, p.pool_rows, p.x_pool,
                                                                     p.x_pool_scale, p.x_planes, p.x_sums, p.hdr);
            break;
        case MOE_A8W8_INT8:
            dispatch_quant_kernel<MOE_A8W8_INT8><<<grid, 256, 0, s>>>(x, p.slot_row, p.T, p.K, p.H, p.pool_rows, p.x_pool,
                                                                      p.x_pool_scale, p.x_planes, p.x_sums, p.hdr);
            break;
        case MOE_A8W4_INT:
            dispatch_quant_kernel<MOE_A8W4_INT><<<grid, 256, 0, s>>>(x, p.slot_row, p.T, p.K, p.H, p.pool_rows, p.x_pool,
                                                                     p.x_pool_scale, p.x_planes, p.x_sums, p.hdr);
            break;
        case MOE_A8W4_FP8_FP4:
            dispatch_quant_kernel<MOE_A8W4_FP8_FP4><<<grid, 256, 0, s>>>(x, p.slot_row, p.T, p.K, p.H, p.pool_rows,
                                                                         p.x_pool, p.x_pool_scale, p.x_planes, p.x_sums, p.hdr);
            break;
        default:  // A16W16: x is already the pool's format
            return launch_dispatch(p, x_bf16, nullptr, s);
    }
    return cudaGetLastError();
}

cudaError_t launch_combine(const Plan& p, uint16_t* y, cudaStream_t s) {
    const int row_vecs = p.H / 8;
    const int64_t n = (int64_t)p.T * row_vecs;
    if (n == 0) return cudaSuccess;
    combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(reinterpret_cast<const uint4*>(p.comb), p.slot_row, p.T,
                                                               p.K, row_vecs, reinterpret_cast<uint4*>(y));
    return cudaGetLastError();
}

cudaError_t launch_debug_wait(const Plan& p, uint64_t timeout_ns, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(p.hdr, 0, sizeof(int32_t) * kHeaderInts, s);
    if (e != cudaSuccess) return e;
    debug_wait_kernel<<<1, 1, 0, s>>>(p.hdr, timeout_ns);
    return cudaGetLastError();
}

cudaError_t launch_expand_gates(const Plan& p, const float* topk_weights, cudaStream_t s) {
    const int n = p.T * p.K;
    if (n == 0) return cudaSuccess;
    expand_gates_kernel<<<(n + 255) / 256, 256, 0, s>>>(topk_weights, n, p.K, p.Kr, p.gates);
    return cudaGetLastError();
}

}  // namespace moe
