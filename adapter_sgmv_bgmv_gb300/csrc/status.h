// Device status codes written to the context's status word, and wait limits.
#pragma once
#include <cstdint>

namespace lora {

// A bounded device wait gives up after this long (nanoseconds of %globaltimer).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

enum DeviceStatus : unsigned {
    kDevOk = 0,
    kDevTimeoutLoad = 1,   // a copy into shared memory did not complete in time
    kDevTimeoutMma = 2,    // a tensor-core commit did not arrive in time
    kDevTimeoutPipe = 3,   // a producer/consumer pipeline slot was not released
    kDevBadShape = 4,      // a kernel found a size it cannot handle (skipped)
    kDevBadId = 5          // a device-resident adapter id the table cannot serve (row skipped)
};

}  // namespace lora
