// replay.cu -- multi-step replay: theta_t = mean_sgd(theta_{t-1}, G_t), then
// m_t = Merkle root of theta_t, for t = 1 .. steps.
//
// "Zoo Per-LLM Chain Soundness" §7 "Reproducibility test plan": start from the
// genesis state, replay each block's gradient batch in chain order with the
// canonical aggregation, then verify H(theta) = m; §4 Theorem
// "Reproducibility" (the per-block update is a deterministic function of the
// pre-state and the batch).  This driver issues, per step, the fixed-order
// mean + SGD kernel and the Merkle commitment of theta on one stream; the
// per-step roots land in device memory so a verifier can compare them with the
// recorded model roots.
#include <vector>

#include "internal.cuh"

using namespace repops;

extern "C" int repops_replay_mean_sgd_commit(int steps, int nC, int64_t len, const float *const *ptrs,
                                             const int *orders, const float *etas, float *theta,
                                             uint32_t leaf, uint8_t *roots_out, cudaStream_t stream) {
    if (steps < 1 || nC < 1 || nC > REPOPS_MEAN_MAX_CONTRIBUTORS || len < 1 || len > INT64_MAX / 4)
        return REPOPS_ERR_INVALID_ARG;
    if (!ptrs || !orders || !etas || !theta || !roots_out) return REPOPS_ERR_INVALID_ARG;
    const uint64_t bytes = uint64_t(len) * 4u;
    // every block is checked before anything runs, so an invalid block cannot
    // leave theta half-replayed
    std::vector<char> seen(static_cast<size_t>(nC));
    for (int t = 0; t < steps; ++t) {
        std::fill(seen.begin(), seen.end(), 0);
        for (int r = 0; r < nC; ++r) {
            const int o = orders[size_t(t) * nC + r];
            if (o < 0 || o >= nC || seen[size_t(o)]) return REPOPS_ERR_ORDER;
            seen[size_t(o)] = 1;
            const float *g = ptrs[size_t(t) * nC + r];
            if (!g) return REPOPS_ERR_INVALID_ARG;
            if (ranges_overlap(theta, bytes, g, bytes)) return REPOPS_ERR_ALIAS;
        }
    }
    if (ranges_overlap(theta, bytes, roots_out, 32u * uint64_t(steps))) return REPOPS_ERR_ALIAS;
    const uint64_t ws_bytes = repops_merkle_workspace_bytes(bytes, leaf);
    if (ws_bytes == 0 && repops_merkle_tree_bytes(bytes, leaf) == 0) return REPOPS_ERR_INVALID_ARG;
    void *ws = nullptr;
    if (ws_bytes > 0) {
        cudaError_t e = scratch_malloc(&ws, ws_bytes, stream);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return REPOPS_ERR_ALLOC;
        }
    }
    int rc = REPOPS_OK;
    for (int t = 0; t < steps && rc == REPOPS_OK; ++t) {
        rc = repops_fixed_order_mean_sgd(nC, len, ptrs + size_t(t) * nC, orders + size_t(t) * nC, etas[t], theta,
                                         stream);
        if (rc == REPOPS_OK)
            rc = repops_merkle_sha256_ws(theta, bytes, leaf, roots_out + 32 * size_t(t), ws, ws_bytes, stream);
    }
    if (ws) {
        cudaError_t e = cudaFreeAsync(ws, stream);
        if (e != cudaSuccess && rc == REPOPS_OK) rc = set_cuda_error(e);
    }
    return rc;
}
