"""CPU oracle for formal-concept enumeration — TEST INFRASTRUCTURE ONLY.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package. The CUDA library never calls it and shares no code with
it; it is the independent definition the library is checked against.

Contents:
  * :func:`cbo`             plain recursive Close-by-One in C (``cbo.c``),
                            single-thread or split over top-level attributes;
  * :func:`cbo_digest`      the same search keeping only an order-independent
                            digest of the intents (for sets too large to hold);
  * :func:`brute_force`     closes every attribute subset (M <= 20) and dedupes;
  * :func:`brute_force_by_objects` derives every object subset (N <= 16);
  * :func:`derive_extent`,
    :func:`derive_intent`   the two derivation operators on packed bitmaps,
                            written with numpy for spot checks at any size;
  * ``lattice``             extents of intents and the cover relation of the concept
                            lattice (``cover_edges``, ``lower_covers_of``), with numpy;
  * ``workcount``           a separate counting pass (``workcount.c``) that counts
                            the algorithmic work of the enumeration in 32-bit
                            words, the numerator of the benchmark's roofline
                            (read from the stored ``tests/golden/work_counts.json``).

Every pin that ties these to the pages' definitions lives in ``tests/``.
"""
from .cbo_binding import build_oracle, cbo, cbo_digest, oracle_library_path  # noqa: F401
from .brute import brute_force, brute_force_by_objects, derive_extent, derive_intent  # noqa: F401
from . import lattice  # noqa: F401
