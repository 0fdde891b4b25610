// Host-side check of the bf16 dispatch ring's load schedule (ring_schedule.h):
// replays the issue / wait order of one CTA for every ring depth, lookahead,
// unit count and failure point, and checks that the drain after a failed wait
// covers exactly the loads that were issued and not yet waited for.  Also
// checks that a stage is never reloaded while an earlier unit's load into it
// may still be unread: the load of unit u is issued only after unit u - NS was
// waited for.  Prints one line; exit code 0 when every case passes.
#include <cstdio>
#include <set>

#include "ring_schedule.h"

using namespace ep;

int main() {
    long cases = 0;
    for (int ns = 2; ns <= 8; ++ns) {
        for (int la = 1; la <= ns - 1; ++la) {
            for (int64_t n = 0; n <= 40; ++n) {
                for (int64_t fail = -1; fail < n; ++fail) {   // -1: no wait fails
                    std::set<int64_t> issued, waited;
                    auto issue = [&](int64_t u) -> bool {
                        if (issued.count(u) || u >= n) return false;
                        if (u >= ns && !waited.count(u - ns)) return false;   // stage still owned
                        issued.insert(u);
                        return true;
                    };
                    for (int64_t u = 0; u < ring_prologue_loads(n, la); ++u) {
                        if (!issue(u)) { std::printf("bad prologue ns=%d la=%d n=%ld\n", ns, la, (long)n); return 1; }
                    }
                    int64_t i = 0;
                    bool failed = false;
                    for (; i < n; ++i) {
                        if (ring_issues_ahead(i, n, la) && !issue(i + la)) {
                            std::printf("bad issue ns=%d la=%d n=%ld i=%ld\n", ns, la, (long)n, (long)i);
                            return 1;
                        }
                        if (!issued.count(i)) {
                            std::printf("wait before load ns=%d la=%d n=%ld i=%ld\n", ns, la, (long)n, (long)i);
                            return 1;
                        }
                        if (i == fail) { failed = true; break; }
                        waited.insert(i);
                    }
                    std::set<int64_t> in_flight;
                    for (int64_t u : issued) if (!waited.count(u)) in_flight.insert(u);
                    std::set<int64_t> drained;
                    if (failed) for (int64_t r = i; r < ring_issued_end(i, n, la); ++r) drained.insert(r);
                    if (in_flight != drained) {
                        std::printf("drain mismatch ns=%d la=%d n=%ld fail=%ld: %zu in flight, %zu drained\n", ns, la,
                                    (long)n, (long)fail, in_flight.size(), drained.size());
                        return 1;
                    }
                    if (!failed && issued.size() != (size_t)n) { std::printf("units not loaded\n"); return 1; }
                    ++cases;
                }
            }
        }
    }
    std::printf("ring schedule ok: %ld cases\n", cases);
    return 0;
}
