// Host-side tag of a launch that uses the forward's dynamic schedule: which
// counter slot of the device array it takes, and the generation number that
// identifies it there.  Plain C++ (no CUDA), so that it can be compiled and
// checked on its own.
#pragma once

#include <cstdint>

namespace attn {

constexpr int kSchedSlots = 256;  // counter slots per device
constexpr int kSchedWords = 4;    // per slot: next unit, CTAs done, owner generation, unused

struct SchedTicket {
    int slot;      // 0 .. kSchedSlots-1
    uint32_t gen;  // nonzero; 0 marks a free slot on the device
};

// Ticket of the n-th launch on a device (n counts from 0).  Slots are taken
// round-robin unless `pinned` is a valid slot index (a testing hook that
// forces launches onto one slot).  The generation is n + 1 modulo 2^32 - 1,
// plus one: it is never 0, and two launches share one only if 2^32 - 1 other
// launches came between them.
inline SchedTicket sched_ticket(uint64_t n, int pinned)
{
    SchedTicket t;
    t.slot = (pinned >= 0 && pinned < kSchedSlots) ? pinned : static_cast<int>(n % kSchedSlots);
    t.gen = static_cast<uint32_t>(n % 0xFFFFFFFFull) + 1u;
    return t;
}

}  // namespace attn
