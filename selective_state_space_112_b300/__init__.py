"""B300-native (sm_103a) Mamba S6 selective-scan forward.

The compute lives in a C-ABI shared library built from ``csrc/``; this
package only marshals arguments to it.
"""
