"""GB300-native wide-beam decode step (libbeamdec) with a thin Python binding.

Importing the package loads nothing; ``beamdec.lib()`` loads the CUDA library
and fails loudly when it has not been built.
"""
