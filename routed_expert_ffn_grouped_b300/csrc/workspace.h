// Host-side layout of the colibri_moe_layer workspace.
#pragma once

#include <stddef.h>

#include "colibri.h"

namespace clb {

// Byte offsets (256-byte aligned) of the layer's intermediates in the workspace.
struct WsLayout {
    size_t err, counters, sync, qx, qx_eo, sx, xc, logits, s, c, offsets, pairs, slots;
    size_t hq, hq_eo, hs, hc, y;
    size_t xbf, hbf;  // prefill (T > DECODE_T_MAX): bf16 codes of x and of q8(h)
    size_t hf;        // decode with 64-element groups: fp32 h rows before their q8
    size_t hpair_count;  // decode with 64-element groups: pair counters in the sync region
    size_t nslots;      // slots at most: the shared expert + min(E, T*K) routed experts
    size_t sync_bytes;  // decode kernel's claim counter, routing counter, (two spare words) |
                        // done_gu [nslots] | done_rb [d/32] | hpair [hpair_count]
    size_t sync_stride; // a layer stack: two such areas sync_stride apart, then the grid
    size_t bar;         // barrier's counter at bar
    size_t sync_end;    // the end of the words zeroed per call (from err)
    size_t fmax, total;
};

constexpr int DECODE_T_MAX = 32;  // larger batches take the tensor-core prefill path

bool cfg_valid(const colibri_layer_cfg *c);
bool uses_gemm(const colibri_layer_cfg *c, int T);
// stack: the workspace of colibri_moe_stack_decode (two control-word areas and a barrier)
WsLayout ws_layout(const colibri_layer_cfg *c, int T, bool stack = false);

}  // namespace clb
