// decode_range.cuh -- the kept-key range of a decode sequence, shared by the
// split kernels (decode.cu) and the one-launch kernel (decode_direct.cu).
#pragma once

namespace attn {

// Range of kept keys of a sequence: [start, end).  The decode query sits at
// position L-1, so the causal mask keeps everything below L; a window keeps
// the W most recent tokens (run.js: kvLen = min(kvLen, W), kvStart = L - kvLen).
__device__ __forceinline__ void seq_range(int L, int cap_eff, int W, int& start, int& end) {
    L = min(max(L, 0), cap_eff);
    start = (W > 0) ? max(0, L - W) : 0;
    end = L;
}

}  // namespace attn
