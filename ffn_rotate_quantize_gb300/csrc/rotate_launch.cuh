// rotate_launch.cuh -- launch helper for rotq_kernel instantiations.
//
// Sizing: a team is one warp when a row needs at most 32 threads (then it
// rotates 32 / (threads per row) rows at once when that divides evenly), else
// the row's threads rounded up to whole warps.  A team's shared memory holds
// its input stages (two when they fit), its transpose tiles (which double as
// the output staging of the bulk store) and a few barriers.  A CTA holds as
// many teams as the thread and shared-memory limits allow; the grid is sized to
// the resident CTAs of the device (persistent teams loop over the rows).
#pragma once

#include "kernels.h"
#include "rotate_fast.cuh"

namespace gbq {

// Resident CTAs per SM of a kernel from its registers (queried once by the caller), threads and
// dynamic shared memory.
inline int resident_ctas(int regs, int threads, size_t smem) {
    const int warp_regs = (regs * 32 + 255) / 256 * 256;
    int per_sm = 65536 / (warp_regs * ((threads + 31) / 32));
    const int by_threads = 2048 / threads;
    const int by_smem = (int)((228 * 1024) / (smem + 1024));
    if (by_threads < per_sm) per_sm = by_threads;
    if (by_smem < per_sm) per_sm = by_smem;
    return per_sm;
}

struct RotqPlan {
    int teams;
    int grid;
    size_t smem;
};

template <int LOGN, int IN, int OUT>
cudaError_t plan_rotq(RotArgs &a, RotqPlan *plan) {
    using Geo = RotGeom<LOGN>;
    constexpr int kMaxSmem = 227 * 1024;
    const int rt = a.G * Geo::TPG;
    const int max_threads = RotqMaxThreads<LOGN>::value;
    const int nin = in_count(IN);
    const int64_t row_in = a.K * in_elem_bytes(IN);
    if (row_in % 16 != 0 || (a.K * out_elem_bytes(OUT)) % 16 != 0) return cudaErrorNotSupported;
    // Rows are moved by bulk copies: every row start must be 16-byte aligned.
    const uintptr_t align = (uintptr_t)a.in0 | (uintptr_t)(a.in1 ? a.in1 : a.in0) | (uintptr_t)a.out;
    if ((align & 15) != 0 || (a.ld_in * in_elem_bytes(IN)) % 16 != 0) return cudaErrorNotSupported;
    a.row_in_bytes = (uint32_t)row_in;
    // Shared memory of a team rotating `rows` rows at once with `stages` input stages.
    auto sizes = [&](int rows, int stages, uint32_t *stage_b, uint32_t *tiles_b) {
        *stage_b = (uint32_t)(((int64_t)rows * nin * row_in + 127) / 128 * 128);
        *tiles_b = (uint32_t)(((int64_t)rows * a.G * Geo::TILE * 8 + 127) / 128 * 128);
        return (int64_t)stages * *stage_b + *tiles_b + kRotMiscBytes;
    };
    if (rt <= 32 && 32 % rt == 0) {
        // Rows pack whole warps: the CTA is one team of W warps that move in lockstep (one
        // instruction stream per SM), W as large as the thread limit and shared memory allow.
        const int rows_per_warp = 32 / rt;
        const int64_t rows_needed = a.M;
        int w = max_threads / 32;
        while (w > 1 && (int64_t)(w - 1) * rows_per_warp >= rows_needed) --w;  // no idle warps for tiny M
        uint32_t sb, tb;
        while (w > 1 && sizes(w * rows_per_warp, 1, &sb, &tb) > kMaxSmem) --w;
        a.team_threads = 32 * w;
        a.rows_per_team = w * rows_per_warp;
    } else if (rt <= 32) {
        a.team_threads = 32;
        a.rows_per_team = 1;
    } else {
        a.team_threads = (rt + 31) / 32 * 32;
        a.rows_per_team = 1;
    }
    if (a.team_threads > max_threads) return cudaErrorNotSupported;
    uint32_t sb, tb;
    a.stages = sizes(a.rows_per_team, 2, &sb, &tb) <= kMaxSmem ? 2 : 1;
    const int64_t tbytes = sizes(a.rows_per_team, a.stages, &sb, &tb);
    if (tbytes > kMaxSmem) return cudaErrorNotSupported;
    a.stage_bytes = sb;
    a.tiles_bytes = tb;
    a.team_bytes = (uint32_t)tbytes;

    int teams = max_threads / a.team_threads;
    const int by_smem = kMaxSmem / (int)a.team_bytes;
    if (by_smem < teams) teams = by_smem;
    if (a.team_threads > 32 && teams > 15) teams = 15;  // named barrier ids 1..15
    const int64_t units = (a.M + a.rows_per_team - 1) / a.rows_per_team;
    if (teams > units) teams = (int)units;
    if (teams < 1) teams = 1;
    plan->teams = teams;
    plan->smem = (size_t)teams * a.team_bytes;

    // Resident CTAs per SM from the kernel's register count (queried once), its threads and shared
    // memory, without an occupancy query on every launch.
    static int regs = -1;  // one per instantiation
    if (regs < 0) {
        cudaError_t e = cudaFuncSetAttribute(rotq_kernel<LOGN, IN, OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kMaxSmem);
        if (e != cudaSuccess) return e;
        cudaFuncAttributes fa{};
        e = cudaFuncGetAttributes(&fa, rotq_kernel<LOGN, IN, OUT>);
        if (e != cudaSuccess) return e;
        regs = fa.numRegs;
    }
    const int per_sm = resident_ctas(regs, teams * a.team_threads, plan->smem);
    if (per_sm < 1) return cudaErrorNotSupported;
    const int64_t ctas_needed = (units + teams - 1) / teams;
    const int64_t resident = (int64_t)per_sm * (a.num_sms > 0 ? a.num_sms : 1);
    plan->grid = (int)(ctas_needed < resident ? ctas_needed : resident);
    return cudaSuccess;
}

// The three-pass kernels (n = 64 or 128, one group per row).
template <int LOGN, int IN, int OUT>
cudaError_t launch_rot_fast(RotArgs a, cudaStream_t st) {
    constexpr int kMaxSmem = 227 * 1024;
    const int nin = in_count(IN);
    const int64_t row_in = a.K * in_elem_bytes(IN);
    const uintptr_t align = (uintptr_t)a.in0 | (uintptr_t)(a.in1 ? a.in1 : a.in0) | (uintptr_t)a.out;
    if ((align & 15) != 0 || (a.ld_in * in_elem_bytes(IN)) % 16 != 0) return cudaErrorNotSupported;
    FastArgs f{};
    a.row_in_bytes = (uint32_t)row_in;
    f.stage_bytes = (uint32_t)((nin * row_in + 127) / 128 * 128);
    int threads;
    auto kern = LOGN == 6 ? rot64_kernel<IN, OUT> : rot128_kernel<IN, OUT>;
    static int regs = -1;  // one per instantiation
    if (regs < 0) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
        if (e != cudaSuccess) return e;
        cudaFuncAttributes fa{};
        e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        regs = fa.numRegs;
    }
    if constexpr (LOGN == 6) {
        threads = 128;
        // Two input stages stream the next row while this one is rotated; when every row fits in
        // the resident CTAs at once with one stage, one stage (more CTAs per SM) is the faster choice.
        const uint32_t tile = (fast_tile_bytes(6) + 127) / 128 * 128;
        const int per_sm1 = resident_ctas(regs, threads, f.stage_bytes + tile + kFastMisc);
        f.stages = (a.M <= (int64_t)per_sm1 * (a.num_sms > 0 ? a.num_sms : 1)) ? 1 : 2;
        f.tile_off = f.stages * f.stage_bytes;
        f.misc_off = f.tile_off + tile;
    } else {
        threads = 512;
        f.stages = 1;
        f.tile_off = 0;  // the tile reuses the stage's memory
        const uint32_t tb = fast_tile_bytes(7);
        f.misc_off = (f.stage_bytes > tb ? f.stage_bytes : (tb + 127) / 128 * 128);
    }
    f.a = a;
    const size_t smem = f.misc_off + kFastMisc;
    if (smem > (size_t)kMaxSmem) return cudaErrorNotSupported;
    const int per_sm = resident_ctas(regs, threads, smem);
    if (per_sm < 1) return cudaErrorNotSupported;
    const int64_t resident = (int64_t)per_sm * (a.num_sms > 0 ? a.num_sms : 1);
    const int grid = (int)(a.M < resident ? a.M : resident);
    if (a.M == 0) return cudaSuccess;
    prof_begin(0, st);
    kern<<<grid, threads, smem, st>>>(f);
    prof_end(st);
    return cudaGetLastError();
}

template <int LOGN, int IN, int OUT>
cudaError_t launch_rotq_t(RotArgs a, cudaStream_t st) {
    if constexpr (LOGN == 6 || LOGN == 7)
        if (a.G == 1) return launch_rot_fast<LOGN, IN, OUT>(a, st);
    RotqPlan plan{};
    cudaError_t e = plan_rotq<LOGN, IN, OUT>(a, &plan);
    if (e != cudaSuccess) return e;
    if (a.M == 0) return cudaSuccess;
    prof_begin(0, st);
    rotq_kernel<LOGN, IN, OUT><<<(unsigned)plan.grid, plan.teams * a.team_threads, plan.smem, st>>>(a);
    prof_end(st);
    return cudaGetLastError();
}

template <int IN, int OUT>
cudaError_t launch_rotq_logn(int logn, RotArgs a, cudaStream_t st) {
    switch (logn) {
        case 4: return launch_rotq_t<4, IN, OUT>(a, st);
        case 5: return launch_rotq_t<5, IN, OUT>(a, st);
        case 6: return launch_rotq_t<6, IN, OUT>(a, st);
        case 7: return launch_rotq_t<7, IN, OUT>(a, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace gbq
