// Host-side size limits shared by the entry points.
//
// Every tensor the kernels index must hold fewer than 2^31 elements: their
// element indices are 32-bit.  A tensor's element count is a product of the
// caller's int dimensions, and such a product can overflow a 64-bit integer
// (four dimensions of 2^16 already reach 2^64).  `within_index_limit` forms
// the product step by step and stops as soon as it passes the limit, so no
// intermediate exceeds 2^62 and no size the caller passes can wrap round
// into an accepted one.
#pragma once

#include <initializer_list>

namespace dcn {

constexpr long long kIndexLimit = (1ll << 31) - 1;

// True when every factor is non-negative and their product is at most
// kIndexLimit.
inline bool within_index_limit(std::initializer_list<long long> factors) {
    long long p = 1;
    for (const long long f : factors) {
        if (f < 0 || f > kIndexLimit) return false;
        p *= f;   // both at most 2^31 - 1: the product fits in 63 bits
        if (p > kIndexLimit) return false;
    }
    return true;
}

}  // namespace dcn
