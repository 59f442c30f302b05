// ssd_plan_check.cpp -- prints the SSD launch plan (ssd_plan.h) for the
// problems given on the command line, one line each:
//   heads nch sms want_seg want_ctas -> dyn seg nseg units ctas
#include <cstdio>
#include <cstdlib>

#include "ssd_plan.h"

int main(int argc, char** argv) {
    for (int i = 1; i + 4 < argc; i += 5) {
        const auto p = ssm::ssdtc::plan(atoll(argv[i]), atoll(argv[i + 1]), atoll(argv[i + 2]),
                                        atoll(argv[i + 3]), atoll(argv[i + 4]));
        std::printf("%d %lld %lld %lld %lld\n", p.dyn ? 1 : 0, p.seg, p.nseg, p.units, p.ctas);
    }
    return 0;
}
