"""GB300-native (sm_103a) blockwise ring attention.

`ops` is the binding of the C-ABI library libra.so (built by `build.build()`);
`inputs` holds the seeded synthetic workloads.  Importing the package does not
load the library; the first call into `ops` does, and fails loudly if the
library is missing.
"""
