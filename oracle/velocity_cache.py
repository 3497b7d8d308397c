"""Conservative DiT velocity-cache schedule, plain Python (test infrastructure only).

Follows the page "perf(minimax-h3): add conservative DiT velocity reuse"
(TeleFuser PR #38), section 3 "Conservative DiT velocity cache": caching is
active only between start_ratio and end_ratio of the denoising process; a DiT
refresh is forced every `refresh_interval`-th step; at most
`max_consecutive_reuse` consecutive steps reuse the previous video/audio
velocity; on a hit the previous DiT-predicted velocities are reused and the
DiT call is skipped.

Readings where the page is silent:
  * progress of step i (0-based) of n is i / n;
  * a reuse needs a velocity computed earlier (never on step 0);
  * "refresh forced every refresh_interval steps" counts steps since the last
    DiT call: a reuse is allowed only while fewer than refresh_interval - 1
    reuses have followed it, and never more than max_consecutive_reuse in a row.
Pinned by the page's own counts: 49 steps -> 34 DiT calls, 15 hits
(tests/golden/velocity_cache_p1.txt).
"""


def schedule(num_steps, start_ratio=0.2, end_ratio=0.8, refresh_interval=2, max_consecutive_reuse=1):
    """List of booleans, True where step i reuses the cached velocity (DiT call skipped)."""
    reuse = []
    have_velocity = False
    run = 0                          # consecutive reuses since the last DiT call
    for i in range(num_steps):
        progress = i / num_steps
        in_window = start_ratio <= progress < end_ratio
        may_reuse = (in_window and have_velocity and run < max_consecutive_reuse
                     and run + 1 < refresh_interval)
        if may_reuse:
            reuse.append(True)
            run += 1
        else:
            reuse.append(False)      # DiT call: fresh velocity, counters restart
            have_velocity = True
            run = 0
    return reuse
