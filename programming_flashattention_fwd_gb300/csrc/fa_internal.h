// fa_internal.h -- declarations shared by the host API (fa_api.cpp) and the kernel
// translation unit (fa_fwd_sm103.cu).  Not part of the public ABI.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Tile sizes: 128 query rows x 128 keys per step (the guide's default block of 128).
constexpr int kBM = 128;
constexpr int kBN = 128;
// Lazy-rescale threshold in log2 units: O and l are rescaled only when the running maximum grows
// by more than tau, so unnormalised p stays <= 2^tau (4096, 16 times below the fp16 maximum).
// Any tau >= 0 gives the same result up to rounding; tau = 0 rescales at every new maximum.
// Each rescale is a round trip of O through registers; with large logits (q, k of std 2) 12
// instead of 8 saved 4 % of the time, and made no difference on unit-variance inputs.
constexpr float kTauDefault = 12.0f;

// Division by a divisor fixed for the launch, as a multiply-high and a shift (numerators below
// 2^31): d, the multiplier m = floor(2^32 (2^l - d) / d) + 1 and the shift l = ceil(log2 d);
// n / d == (umulhi(n, m) + n) >> l.  Filled on the host (make_fastdiv in schedule.h).
struct FastDiv {
    uint32_t d, mul, shr;
};

// Per-launch scalar parameters (passed by value to the kernel).
struct Params {
    void *o;            // [B, Hq, Sq, D] 16-bit
    float *lse;         // [B, Hq, Sq] fp32
    int B, Hq, Hkv, Sq, Sk;
    int Tq, Tk;         // number of 128-row query / key tiles
    int NP;             // query-tile pairs per (b, hq): ceil(Tq / 2)
    int group;          // Hq / Hkv
    int num_units;      // work units (query-tile pairs) in the whole problem: B * Hq * NP
    float sl2;          // |scale| * log2(e): the exp2-domain multiplier of the scores
    uint32_t smode;     // 0: scale > 0; 1: scale < 0 (scores negated); 2: scale == 0 (scores zeroed)
    int coff;           // causal offset: key j allowed for query i iff j <= i + coff (0 top-left, Sk - Sq bottom-right)
    uint64_t timeout_ns;// watchdog limit of each bounded wait
    uint32_t inject;    // fault-injection mask (0 in normal use)
    uint32_t o_al32;    // o is 32-byte aligned: output rows are written in full 32-byte sectors
    float tau;          // lazy-rescale threshold (kTauDefault outside tests)
    // the schedule's divisors (set_schedule_divisors in schedule.h): B*Hq, NP, Tq, Hq, Hq/Hkv
    FastDiv f_nbh, f_np, f_tq, f_hq, f_group;
};

// The TMA descriptors: q, k, v, o as 3-D (D, S, B*H) tensors, 64 x 128 boxes, 128B swizzle
// (o: the two-tile kernel writes tile b's output rows with bulk tensor stores).
struct Maps {
    CUtensorMap q, k, v, o;
};

// Checks shared by the entry points, made before any CUDA call: the argument checks of
// fa_fwd (returns FA_OK for a valid or empty problem, else the fa_status_t code), and
// "the current device is an sm_103 part" (cached per device).
int check_fwd_args(const void *q, const void *k, const void *v, const void *o, const float *lse, int B, int Hq,
                   int Hkv, int Sq, int Sk, int D, int causal, float scale, int kernel);
int check_device();

// Launches the forward kernel for (D, dtype, causal).  Returns the cudaGetLastError() of the launch.
cudaError_t launch_fwd(int D, bool bf16, bool causal, const Maps &maps, const Params &p, cudaStream_t stream);

// Reads and clears the current device's watchdog word (synchronous on `stream`).
cudaError_t read_and_clear_status(cudaStream_t stream, uint32_t *word);

// One query tile per CTA, 64-key steps, double-buffered scores (D = 64, 128 or 256).  K/V maps
// use 64-row boxes; Params.Tk counts 64-key tiles and num_units = B * Hq * Tq.
cudaError_t launch_fwd1(int D, int keys, bool bf16, bool causal, const Maps &maps, const Params &p,
                        cudaStream_t stream);   // keys per step: 64 (D 64 / 128 / 256) or 128 (D 128)
cudaError_t read_and_clear_fa1_status(uint32_t *word);

// ---------------------------------------------------------------- tiled matrix product
struct GemmParams {
    void *c;               // [M, N] row-major, 16-bit (input type) or fp32
    const float *bias;     // [N] fp32, or nullptr when the epilogue has no bias
    int M, N, K;
    int Tm, Tn, nK;        // 128-row tiles, 256-column tiles, 64-wide K blocks
    int num_tiles;         // Tm * Tn
    uint64_t timeout_ns;
};
// epilogue: 0 none, 1 + bias, 2 tanh-GELU(. + bias).  A map: 2-D (K, M), box 64 x 128;
// B map: 2-D (N, K), box 64 x 64; both 128B swizzle.
cudaError_t launch_gemm(bool bf16, bool out_f32, int epilogue, const CUtensorMap &a, const CUtensorMap &b,
                        const GemmParams &p, cudaStream_t stream);
cudaError_t read_and_clear_gemm_status(uint32_t *word);

// ---------------------------------------------------------------- row softmax
// x, y: [rows, cols] row-major, fp32 or bf16 (same type); one launch, any cols >= 1.
cudaError_t launch_softmax_rows(bool bf16, const void *x, void *y, int rows, int cols, cudaStream_t stream);
cudaError_t read_and_clear_softmax_status(uint32_t *word);

} // namespace fa
