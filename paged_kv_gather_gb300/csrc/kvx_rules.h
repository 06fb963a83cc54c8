// kvx_rules.h -- launch-shape rules the host applies before a launch, kept in one place so
// that the launch path and the public query (kvx_roundtrip_unit, for the time model) agree.
#pragma once

#include <stdint.h>

#include "../../include/kvx.h"

namespace kvx {

// Units of a round trip (kvx_roundtrip_chunks): `batch` page segments per unit, or, with
// slices > 1, one row slice of a segment per unit (slices per segment); `sm_cap` is the SM
// cap the launch uses.
struct RoundTripRule {
    int32_t batch;
    int32_t slices;
    int32_t sm_cap;
};

// The rule for page segments of page_size rows of token_bytes.  user_cfg: whether the caller
// gave a configuration (without one, short segments get more SMs); sm_cap and batch: the
// resolved configuration's (0 = every SM, 0 = automatic); num_sms: the device's SM count.
RoundTripRule roundtrip_rule(int32_t page_size, int64_t token_bytes, bool user_cfg,
                             int32_t sm_cap, int32_t batch, int num_sms);

}  // namespace kvx
